"""Oracle for the low-rank bottleneck block (TEST INFRASTRUCTURE ONLY).

A plain, slow, fp64 CPU restatement of what the BOOST pages describe
("BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank Large
Language Models", arXiv 2512.12131, technical summary §2.1-§2.2). It exists to
prove the CUDA path right and to give the CPU baseline a number.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it. The product path (``rank_bottleneck_online_gb300``) never
imports, calls or links anything here, and nothing here imports the product
path: the two share no code. The only shared module is the seeded input
generator ``rank_bottleneck_online_gb300.inputs``, which holds none of the
method's arithmetic.

Parity status: every function is pinned by a ``-m "not gpu"`` test (closed
forms, library routines, finite differences, brute force); none is
"parity unpinned".
"""

from .bottleneck import (  # noqa: F401
    BF16_MAX,
    to_bf16,
    silu,
    silu_grad,
    identity,
    identity_grad,
    act_fns,
    shard_bounds,
    group_bounds,
    exchange_elems,
    rmsnorm_stats,
    btp_shard_partials,
    btp_reduce,
    block_fwd_reference,
    block_bwd_reference,
    block_fwd,
    block_bwd,
    swiglu_fwd,
    swiglu_bwd,
    mlp_fwd,
    mlp_bwd,
    layer_fwd,
    layer_bwd,
    svd_pair_fwd,
    svd_pair_bwd,
    rel_errors,
)
