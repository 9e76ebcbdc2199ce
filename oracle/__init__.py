"""Plain, slow, fp64 CPU oracle of the fused MoE expert forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) may import, call or link anything under ``oracle/``; only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) use it.  It shares no code, tables or helpers with the
CUDA path.

What it computes (the page "fused_moe.py 分析", §1.1-1.4, and the page
"Blackwell 上的 DeepGEMM FusedMoE（vLLM）", §2.6):

    y_t = sum_{i : id[t,i] >= 0} w[t,i] * W2_e( SiLU(W1gate_e x_t) * (W1up_e x_t) ),
    e = id[t,i],

organised in the five stages of the pages: block-aligned routing and permute,
grouped GEMM1, SiLU-and-mul (optionally dynamic FP8 quantisation), grouped
GEMM2, weighted unpermute with a top-k reduce.  Arithmetic is fp64; the values
are rounded only where the data path stores them in a narrower type (bf16
GEMM outputs, e4m3 codes with fp32/UE8M0 scales).

Modules:
  codecs   -- bf16 / fp32 rounding, e4m3fn, E2M1, E8M0 codecs.
  routing  -- moe_align_block_size (counting sort with block padding), the
              M_sum bound, inverse permutation.
  experts  -- permute, activation quantisation, grouped GEMMs, SiLU-and-mul,
              unpermute-reduce, the whole forward (permuted form) and the
              per-token brute-force form.
  router   -- the step before the path: softmax / sigmoid scores, top-k
              selection, renormalisation and the expert-parallel expert map.

Every function has a pin in ``tests/test_oracle_*.py`` (library routines,
closed forms, invariants, brute force, hand-worked fixtures); none is marked
"parity unpinned".
"""
from . import codecs, routing, experts, router  # noqa: F401
