"""Emulation of limited-precision accumulation in an FP8 GEMM (a context study).

Test infrastructure, like the rest of oracle/: only tests and the bench's CPU
leg use it; the CUDA path never does.

The pages say that on H800 the tensor cores accumulate FP8 products keeping
only about 14 bits (dssusan.co.kr post 91437, paragraph 2), by fixed-point
accumulation that first aligns the mantissas of the products by shifting right
to the largest exponent ("Deepseek - Not For everyone", paragraph 5). They
also say that for K = 4096 this gives a maximum relative error of nearly 2 %
(dssusan post, paragraph 4), and that copying partial sums to FP32 registers at
a fixed K interval cures it (same post, paragraph 3).  The hardware's order
and rounding are not given; this module takes the plainest reading of those
sentences:

  * the products a_k * b_k are exact (FP8 x FP8 fits a double) and are added
    one at a time in k order;
  * before each addition, the running sum and the product are both truncated
    toward zero onto the grid 2^(E - (bits - 1)), E being the larger of their
    binary exponents: right-shift alignment that keeps `bits` bits of the
    larger operand; the aligned values are then added exactly;
  * with promotion every n_c products, the limited partial sum is added to an
    FP32 accumulator (one round-to-nearest FP32 addition) and restarted.

Parity unpinned against hardware: there are no H800 measurements here.  The
tests pin the emulator against closed forms instead (unlimited bits give the
exact sequential sum; promotion after every product gives the FP32 sequential
sum; hand-worked truncation and swamping cases).
"""
import numpy as np


def _trunc_to_grid(x: np.ndarray, ulp: np.ndarray) -> np.ndarray:
    # x / ulp and the product back are exact: ulp is a power of two
    return np.trunc(x / ulp) * ulp


def add_aligned(s, p, bits: int):
    """One addition of the limited-precision accumulator, element-wise."""
    s = np.asarray(s, np.float64)
    p = np.asarray(p, np.float64)
    m = np.maximum(np.abs(s), np.abs(p))
    _, e = np.frexp(np.where(m > 0, m, 1.0))  # m = f * 2^e, f in [0.5, 1): exponent E = e - 1
    ulp = np.ldexp(1.0, (e - 1) - (bits - 1))
    out = _trunc_to_grid(s, ulp) + _trunc_to_grid(p, ulp)
    return np.where(m > 0, out, 0.0)


def limited_acc_dot(a, b, bits: int, n_c=None) -> np.ndarray:
    """Row-wise dot products sum_k a[r, k] * b[r, k] with the accumulator above.

    a, b: [R][K] arrays of exactly representable values (e.g. dequantised
    E4M3 codes).  n_c: promotion interval in products (None: never promote;
    the whole K is accumulated at limited precision)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    R, K = a.shape
    part = np.zeros(R)
    acc32 = np.zeros(R, np.float32)
    for k in range(K):
        part = add_aligned(part, a[:, k] * b[:, k], bits)
        if n_c is not None and ((k + 1) % n_c == 0 or k == K - 1):
            # the partial has at most `bits` + 1 significant bits: exact in FP32 for bits <= 23
            acc32 = np.float32(acc32) + part.astype(np.float32)
            part = np.zeros(R)
    return part if n_c is None else acc32.astype(np.float64)
