"""GB300-native low-rank bottleneck block (BOOST, arXiv 2512.12131).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/boost_block.h``). ``binding`` loads
it through ctypes and marshals torch tensors to raw device pointers; ``block``
composes the C-ABI calls into the workloads (one block, the LLaMA MLP, the
full layer, the SVD pair). ``inputs`` draws the seeded synthetic tensors.

Importing this package does not load the library; ``binding.lib()`` does,
and raises if the library has not been built.
"""

__all__ = ["inputs", "binding", "block", "build"]
