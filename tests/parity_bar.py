"""The parity bar of the GPU tests and the oracle's process pool.

NVFP4 path, against the tile-by-tile SA3 emulation (the same Bc = 128, the
oracle's own quantiser):
  |O_gpu - O_emul| <= NVFP4_TOL * max|O_emul| + B
where B is the oracle's decision-ambiguity bound: a P quantisation decision
whose input lies within TIE_REL (relative) of an e2m1/e4m3 rounding boundary
may go either way (the kernel forms P2 from float32 tensor-core scores and
ex2.approx, the oracle from exact products; several results are correct
there), and B is the most any of them can move O.  TIE_REL comes from the
measured score error of the kernel's own S step plus the arithmetic rounding
of the exponent path (tests/test_gpu_score_error.py derives the bound and
checks that TIE_REL covers it with margin without being far wider).  Rows
whose decisions are all unambiguous meet CLEAN_TOL * max|O_emul| (there the
two sides quantise P identically and differ only by float32 accumulation
order and the exponentials of the row sum and rescaling).  Checked on the
FP32 output (SA_OUT_FP32); the bf16 output adds its own rounding (2^-9 of
each element).  The cosine to exact FP64 attention must not fall below the
emulation's own cosine by more than COS_SLACK (the scheme, not the kernel,
sets that cosine: about 0.98 on these inputs, below the 0.995 target).

BF16 path: mean per-head cosine >= BF16_COS against exact FP64 attention and
max-abs <= BF16_TOL * max|O| (bf16 rounding of P and of O, 2^-9 relative each).
"""

import atexit
import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

NVFP4_TOL = 2e-3
TIE_REL = 2e-5
# The smooth-Q variant adds the float32 score correction dS before the
# softmax: its error, (D/16 + 17) * 2^-24 * sum_c |qbar_c K^'_jc| (the FMA
# chains of smooth_q.cu), and the rounding of S + dS widen the decision
# window; tests/test_gpu_smooth_q.py checks that TIE_REL_SQ - TIE_REL covers
# twice that extra relative error on every smooth-Q parity case.
TIE_REL_SQ = 4e-5
CLEAN_TOL = 1e-5
COS_SLACK = 2e-3
BF16_COS = 0.99999
BF16_TOL = 8e-3

_pool = None


def oracle_pool():
    """A process pool for per-head oracle work, started with spawn (a pool
    forked after the first GPU call would inherit a CUDA context)."""
    global _pool
    if _pool is None:
        n = max(1, min(8, (os.cpu_count() or 2) // 2))
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(var, "2")
        _pool = ProcessPoolExecutor(max_workers=n, mp_context=multiprocessing.get_context("spawn"))
        atexit.register(_pool.shutdown)
    return _pool


def head_oracle(args):
    """Exact FP64 attention of one head at the given rows and, for the NVFP4
    path (mode "nvfp4", or "nvfp4_sq" for the smooth-Q variant's operands),
    the SA3 emulation with its decision-ambiguity bound (runs in a pool
    worker).  q [1,1,Lq,d], k and v [1,1,Lkv,d] float32 (the head's kv head)."""
    q, k, v, causal, rows, mode, tie_rel = args
    from oracle import attention as A
    ex = A.exact_attention(q, k, v, causal, rows=rows)[0, 0]
    if mode not in ("nvfp4", "nvfp4_sq"):
        return ex, None, None
    if mode == "nvfp4_sq":
        (qd, kd, vd), _ = A.dequantized_operands_sq(q, k, v)
    else:
        (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
    em, bd = A.sa3_emulated_attention(qd, kd, vd, causal, rows=rows, tie_rel=tie_rel, return_bound=True)
    return ex, em[0, 0], bd[0, 0]
