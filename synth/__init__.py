"""Seeded synthetic inputs, reproducible bit for bit on the host and on the GPU.

This module generates data only: it holds none of the MoE layer's arithmetic.
Both the oracle (on the host) and the CUDA path (through ``synth/libsynth.so``)
take their inputs from the one generator defined here, so that the two sides
see identical bytes without copying tens of gigabytes of weights across.

Generator (counter based, stateless):

* A tensor is identified by ``(seed, tensor_id)``.  Its key is
  ``mix64((seed * GAMMA + tensor_id) mod 2**64)``.
* Element ``i`` draws four 64-bit words ``mix64(key + (4*i + j + 1) * GAMMA)``
  for ``j = 0..3``: the SplitMix64 output sequence of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014) started at
  state ``key`` and advanced to position ``4*i + j + 1``.
* Normal draws: each word gives three 21-bit fields (bits 0-20, 21-41, 42-62);
  the twelve fields ``u_1..u_12`` of the four words are summed (the Irwin-Hall
  construction of an approximately standard normal variate, sum of twelve
  uniforms minus six) as ``n = (sum(u) - 6*(2**21 - 1)) * 2**-21``.  Every step
  is exact in float32 (``|sum - 6*(2**21-1)| < 2**24``), so host and device
  agree bit for bit.  The value is then ``fl32(n * sigma)`` (one IEEE float32
  multiply) and, for bfloat16 tensors, rounded to nearest-even in bfloat16.
  The law has mean 0 and variance 1 exactly (before the scale) and is bounded
  at +-6 standard deviations.
* Uniform draws on ``[lo, lo + width)``: ``t = ((w0 >> 40) + 0.5) * 2**-24`` from
  the first word, then ``fl32(lo + width * t)`` evaluated in float64 with one
  rounding per operation (no fused multiply-add), then rounded to float32.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_FIELD_MASK = (1 << 21) - 1
_NORMAL_BIAS = 6 * _FIELD_MASK          # 6 * (2**21 - 1): mean of the 12-field sum
_NORMAL_SCALE = np.float32(2.0 ** -21)

# Tensor identifiers of the layer's inputs (stable across releases: changing
# one changes every stored expected value written from these inputs).
TID_X = 1          # activations x [T, h]
TID_WR = 2         # router weight [E, h]
TID_W13 = 3        # expert gate/up weights [E, 2I, h]
TID_W2 = 4         # expert down weights [E, h, I]
TID_SEL_BIAS = 5   # per-expert selection bias [E]
TID_ZIPF = 6       # surrogate logits used to fit the Zipf logit offsets
TID_W13S = 7       # shared expert gate/up weights [2*shared_I, h]
TID_W2S = 8        # shared expert down weights [h, shared_I]
TID_TEST = 100     # first id free for test-only tensors


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2**64)."""
    z &= MASK64
    z ^= z >> 30
    z = (z * _M1) & MASK64
    z ^= z >> 27
    z = (z * _M2) & MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def tensor_key(seed: int, tensor_id: int) -> int:
    return mix64_int((seed * GAMMA + tensor_id) & MASK64)


def words(seed: int, tensor_id: int, index: np.ndarray, j: int) -> np.ndarray:
    """Word ``j`` (0..3) of the elements at ``index`` (int64 array)."""
    key = np.uint64(tensor_key(seed, tensor_id))
    with np.errstate(over="ignore"):
        ctr = index.astype(np.uint64) * np.uint64(4) + np.uint64(j + 1)
        return _mix64(key + ctr * np.uint64(GAMMA))


def _normal_f32(seed: int, tensor_id: int, index: np.ndarray, sigma: np.float32) -> np.ndarray:
    s = np.zeros(index.shape, dtype=np.int64)
    m = np.uint64(_FIELD_MASK)
    for j in range(4):
        w = words(seed, tensor_id, index, j)
        s += (w & m).astype(np.int64)
        s += ((w >> np.uint64(21)) & m).astype(np.int64)
        s += ((w >> np.uint64(42)) & m).astype(np.int64)
    n = (s - _NORMAL_BIAS).astype(np.float32) * _NORMAL_SCALE   # exact
    return n * np.float32(sigma)                                   # one IEEE fp32 multiply


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, nearest-even, returned as uint16 bit patterns."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_at(seed: int, tensor_id: int, index, sigma: float, dtype: str, chunk: int = 1 << 22) -> np.ndarray:
    """Normal draws at flat element indices.  Returns float32 ('f32') or uint16 bf16 bits ('bf16')."""
    index = np.asarray(index, dtype=np.int64).reshape(-1)
    sig = np.float32(sigma)
    out = np.empty(index.shape, dtype=np.float32 if dtype == "f32" else np.uint16)
    for a in range(0, index.size, chunk):
        v = _normal_f32(seed, tensor_id, index[a:a + chunk], sig)
        out[a:a + chunk] = v if dtype == "f32" else f32_to_bf16_bits(v)
    return out


def _host_lib():
    """The C host generator (synth/libsynth_host.so), or None if not built."""
    global _HOST
    if _HOST is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth_host.so")
        if not os.path.exists(path):
            return None
        lib = ctypes.CDLL(path)
        lib.synth_host_fill_normal.restype = None
        lib.synth_host_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_int64, ctypes.c_float]
        _HOST = lib
    return _HOST


_HOST = None


def normal(seed: int, tensor_id: int, shape, sigma: float, dtype: str, start: int = 0,
           use_c: bool = True) -> np.ndarray:
    """A whole tensor (or a contiguous slice of one starting at flat element ``start``).

    Uses the C host generator when it is built (same values, many times faster)."""
    n = int(np.prod(shape))
    lib = _host_lib() if use_c else None
    if lib is None:
        return normal_at(seed, tensor_id, np.arange(start, start + n, dtype=np.int64), sigma, dtype).reshape(shape)
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    lib.synth_host_fill_normal(out.ctypes.data, n, 0 if dtype == "f32" else 1, seed, tensor_id, start,
                               float(np.float32(sigma)))
    return out.reshape(shape)


def uniform(seed: int, tensor_id: int, n: int, lo: float, hi: float) -> np.ndarray:
    """float32 draws on [lo, hi)."""
    idx = np.arange(n, dtype=np.int64)
    w = words(seed, tensor_id, idx, 0)
    t = ((w >> np.uint64(40)).astype(np.float64) + 0.5) * 2.0 ** -24
    width = float(hi) - float(lo)
    return (float(lo) + width * t).astype(np.float32)


def uniform_topk_ids(seed: int, tensor_id: int, T: int, E: int, K: int) -> np.ndarray:
    """Uniformly random K-subsets of the E experts for each of T tokens (int32 [T, K]).

    Each (token, expert) pair gets an iid 64-bit word; the K experts with the
    smallest words form a uniformly random subset.  Used only to build
    routing-free workloads (balls-into-bins), never by the layer itself.
    """
    idx = np.arange(T * E, dtype=np.int64)
    w = words(seed, tensor_id, idx, 0).reshape(T, E)
    return np.argsort(w, axis=1, kind="stable")[:, :K].astype(np.int32)


def zipf_logit_offsets(seed: int, E: int, s: float = 1.1, n_rows: int = 1 << 16, iters: int = 100) -> np.ndarray:
    """Per-expert logit offsets o[e] so that argmax_e (z_e + o_e), z ~ N(0, I_E), lands on
    expert e with probability p_e proportional to (e+1)**-s.

    Fixed-point fit: start at o = log p; repeat o <- o + 0.5 (log p - log q), where q
    is the empirical argmax frequency over ``n_rows`` seeded standard-normal rows.
    Router logits x W_r with x ~ N(0,1) and W_r ~ N(0, 1/h) are approximately
    N(0, I_E), so the surrogate rows stand in for them.  Returns float32 [E].
    """
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    z = normal(seed, TID_ZIPF, (n_rows, E), 1.0, "f32").astype(np.float64)
    o = np.log(p)
    for _ in range(iters):
        hits = np.bincount(np.argmax(z + o, axis=1), minlength=E).astype(np.float64)
        q = np.maximum(hits, 0.5) / n_rows
        o = o + 0.5 * (np.log(p) - np.log(q))
        o -= o.max()
    return o.astype(np.float32)
