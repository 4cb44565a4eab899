"""Seeded synthetic decode and prefill workloads.

Every array is drawn from numpy's PCG64 ``default_rng(seed)`` as N(0,1) in
fp32 and, for bf16 workloads, rounded to bf16 (round to nearest even) and kept
as raw uint16 bit patterns.  Layouts are "bshd": queries ``[B, T_q, H_q, D]``
(decode) or ``[B, S, H_q, D]`` (prefill), keys and values ``[B, T, H_kv, D]``.

The planted structure follows the workloads the pages measure on (passkey
style needles for decode in the InfiniteHiP summary, vertical columns and
slash diagonals for the MInference vertical-slash heads); the datasets
themselves are not used.  Nothing here scores, selects or normalises anything.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 24  # elements drawn per call, keeps fp32 temporaries bounded


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to FP8 E4M3 (nearest, ties to even, saturating at +-448);
    return uint8 codes.  Positive codes grow with the value (code = 8 * biased exponent
    + mantissa, subnormals m * 2^-9 below 2^-6), so the rounding is done on the code."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))
    E = ex.astype(np.int64) - 1                       # floor(log2 a) for a >= 2^-6
    normal = np.rint(a / np.exp2(E - 3.0)).astype(np.int64) + 8 * E + 48
    sub = np.rint(a * 512.0).astype(np.int64)         # a < 2^-6: multiples of 2^-9
    code = np.where(a < 2.0 ** -6, sub, normal)
    code = np.minimum(code, 126)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def with_fp8_kv(case: "DecodeCase") -> "DecodeCase":
    """The same decode case with its keys and values stored as FP8 E4M3 (rounded from
    their bf16 / fp32 values); the queries keep their type."""
    from dataclasses import replace
    src = case.dtype == "bf16"
    k = f32_to_e4m3_bits(_as_f32(case.k, src))
    v = f32_to_e4m3_bits(_as_f32(case.v, src))
    return replace(case, name=case.name + "_fp8kv", k=k, v=v, kv_dtype="e4m3")


def _normal_bits(rng: np.random.Generator, shape, bf16: bool) -> np.ndarray:
    """Draw N(0,1) fp32 in fixed-size pieces; bf16 bits or fp32 values."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        piece = rng.standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = f32_to_bf16_bits(piece) if bf16 else piece
    return out.reshape(shape)


def _as_f32(a: np.ndarray, bf16: bool) -> np.ndarray:
    if not bf16:
        return a.astype(np.float32)
    return (a.astype(np.uint32) << 16).view(np.float32)


def _store(a32: np.ndarray, bf16: bool) -> np.ndarray:
    return f32_to_bf16_bits(a32) if bf16 else a32.astype(np.float32)


@dataclass
class DecodeCase:
    """One batched decode step: queries, a resident KV cache and the selection knobs."""

    name: str
    B: int
    T_max: int
    T_q: int
    H_q: int
    H_kv: int
    D: int
    dtype: str                     # "bf16" (uint16 bits) or "f32"
    chunk: tuple                   # l_c per pruning stage
    keep: tuple                    # k (tokens) per pruning stage
    n_sink: int
    n_stream: int
    kv_len: np.ndarray             # int32 [B]
    q: np.ndarray                  # [B, T_q, H_q, D]
    k: np.ndarray                  # [B, T_max, H_kv, D]
    v: np.ndarray                  # [B, T_max, H_kv, D]
    planted: list = field(default_factory=list)  # per batch row: planted key positions
    kv_dtype: str = ""             # "" (as dtype) or "e4m3" (uint8 codes) for k and v

    @property
    def kvd(self) -> str:
        """Storage type of k and v."""
        return self.kv_dtype or self.dtype

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


@dataclass
class PrefillCase:
    """One causal prefill: Q/K/V for the whole prompt and the vertical-slash budgets."""

    name: str
    B: int
    S: int
    H_q: int
    H_kv: int
    D: int
    last_q: int
    n_vertical: int
    n_slash: int
    q: np.ndarray                  # bf16 bits [B, S, H_q, D]
    k: np.ndarray                  # bf16 bits [B, S, H_kv, D]
    v: np.ndarray                  # bf16 bits [B, S, H_kv, D]
    planted_columns: np.ndarray    # key positions given a shared direction with the queries
    planted_offsets: np.ndarray    # query-minus-key offsets given a shared positional code
    block: int = 64

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


# --------------------------------------------------------------------------- decode

def decode_case(name, *, B, T, T_q, H_q, H_kv, D, dtype, chunk, keep, n_sink, n_stream,
                seed, plant="uniform", n_plant=64, kv_len=None, noise=0.5,
                seeds_per_row=None) -> DecodeCase:
    """Generic decode workload.

    ``plant`` chooses where keys that resemble a query are placed inside the
    candidate range [n_sink, T - n_stream):
      * "uniform": ``n_plant`` distinct uniform positions per KV head g, key
        K[p, g] = Q[0, h] + noise*N(0,1) with h = G*g + (j mod G);
      * "spread": ``n_plant`` positions spread evenly, shared by all KV heads;
      * "cluster": one contiguous run of ``n_plant`` tokens at a random offset;
      * "rows": (single head, T_q rows) K[p_i] = Q[t_i] + noise*N(0,1), t_i = i;
      * "none".
    ``seeds_per_row`` gives each batch row its own generator (batch workloads).
    """
    bf16 = dtype == "bf16"
    G = H_q // H_kv
    kv_len = np.full(B, T, dtype=np.int32) if kv_len is None else np.asarray(kv_len, np.int32)
    q = np.empty((B, T_q, H_q, D), np.uint16 if bf16 else np.float32)
    k = np.empty((B, T, H_kv, D), q.dtype)
    v = np.empty((B, T, H_kv, D), q.dtype)
    planted = []
    shared = np.random.default_rng(seed)
    for b in range(B):
        rng = shared if seeds_per_row is None else np.random.default_rng(seeds_per_row[b])
        q[b] = _normal_bits(rng, (T_q, H_q, D), bf16)
        k[b] = _normal_bits(rng, (T, H_kv, D), bf16)
        v[b] = _normal_bits(rng, (T, H_kv, D), bf16)
        Tb = int(kv_len[b])
        lo, hi = n_sink, max(n_sink, Tb - n_stream)
        rows = []
        if plant != "none" and hi - lo >= n_plant:
            qf = _as_f32(q[b], bf16)
            if plant == "rows":
                pos = np.sort(rng.choice(np.arange(lo, hi), size=n_plant, replace=False))
                for i, p in enumerate(pos):
                    t = i % T_q
                    for g in range(H_kv):
                        kv = qf[t, G * g] + noise * rng.standard_normal(D, dtype=np.float32)
                        k[b, p, g] = _store(kv, bf16)
                rows = [int(p) for p in pos]
            else:
                if plant == "uniform":
                    per_g = [np.sort(rng.choice(np.arange(lo, hi), size=n_plant, replace=False))
                             for _ in range(H_kv)]
                elif plant == "spread":
                    n0 = hi - lo
                    pos = lo + ((np.arange(n_plant) + 0.5) * n0 / n_plant).astype(np.int64)
                    per_g = [pos] * H_kv
                elif plant == "cluster":
                    start = int(rng.integers(lo, hi - n_plant + 1))
                    per_g = [np.arange(start, start + n_plant)] * H_kv
                else:
                    raise ValueError(plant)
                for g in range(H_kv):
                    for j, p in enumerate(per_g[g]):
                        h = G * g + (j % G)
                        kv = qf[0, h] + noise * rng.standard_normal(D, dtype=np.float32)
                        k[b, p, g] = _store(kv, bf16)
                rows = sorted({int(p) for pg in per_g for p in pg})
        planted.append(rows)
    return DecodeCase(name, B, T, T_q, H_q, H_kv, D, dtype, tuple(chunk), tuple(keep),
                      n_sink, n_stream, kv_len, q, k, v, planted)


def decode_tiny() -> DecodeCase:
    """1 query head / 1 KV head, d=64, fp32, T=2048, 32 query rows, 8 planted keys, seed 0."""
    return decode_case("decode_tiny_T2048_d64_f32", B=1, T=2048, T_q=32, H_q=1, H_kv=1, D=64,
                       dtype="f32", chunk=(64, 16, 4), keep=(1024, 256, 128), n_sink=16,
                       n_stream=64, seed=0, plant="rows", n_plant=8)


def decode_128k() -> DecodeCase:
    """Llama-3-8B-shaped GQA decode (32q/8kv, d=128, bf16), context 131072, seed 1."""
    return decode_case("decode_gqa_T131072", B=1, T=131072, T_q=1, H_q=32, H_kv=8, D=128,
                       dtype="bf16", chunk=(256, 64, 16, 4), keep=(32768, 16384, 8192, 4096),
                       n_sink=128, n_stream=1024, seed=1, plant="uniform", n_plant=64)


def decode_1m() -> DecodeCase:
    """Same GQA shape at context 1,048,576 with 256 evenly spread needles, seed 2."""
    return decode_case("decode_gqa_T1048576", B=1, T=1 << 20, T_q=1, H_q=32, H_kv=8, D=128,
                       dtype="bf16", chunk=(256, 64, 16, 4), keep=(32768, 16384, 8192, 4096),
                       n_sink=128, n_stream=1024, seed=2, plant="spread", n_plant=256)


def decode_batch16() -> DecodeCase:
    """Batch 16 at context 32768, one planted 64-token cluster per sequence, seeds 300+b."""
    return decode_case("decode_gqa_B16_T32768", B=16, T=32768, T_q=1, H_q=32, H_kv=8, D=128,
                       dtype="bf16", chunk=(256, 64, 16, 4), keep=(16384, 8192, 4096, 2048),
                       n_sink=64, n_stream=512, seed=300, plant="cluster", n_plant=64,
                       seeds_per_row=[300 + b for b in range(16)])


def decode_steps(case: DecodeCase, n_steps: int, seed: int, drift: float = 0.3):
    """A seeded decoding loop over one case: per step s a query block
    q_s = case.q + drift * N(0,1) (rounded to the case's storage type) and kv_len_s =
    min(case.kv_len + s, T_max), i.e. one new token per step in every row.  Returns a
    list of (q_s, kv_len_s); step 0 uses case.q itself."""
    bf16 = case.dtype == "bf16"
    rng = np.random.default_rng(seed)
    base = _as_f32(case.q, bf16)
    out = []
    for s in range(n_steps):
        if s == 0:
            q = case.q.copy()
        else:
            q = _store(base + drift * rng.standard_normal(base.shape, dtype=np.float32), bf16)
        kv = np.minimum(case.kv_len.astype(np.int64) + s, case.T_max).astype(np.int32)
        out.append((q, kv))
    return out


# --------------------------------------------------------------------------- prefill

def prefill_case(name, *, B=1, S, H_q, H_kv, D, seed, last_q=64, n_vertical=1000,
                 n_slash=6096, n_columns=16, n_far_offsets=4, near_offsets=65,
                 beta=4.0, alpha=4.0, col_q=3.0, col_k=12.0) -> PrefillCase:
    """Causal prefill with planted vertical columns and slash diagonals.

    Columns: ``n_columns`` distinct key positions j_v; per KV head g a random
    unit direction e_g is added to every query of the group (``col_q``) and to
    K[j_v, g] (``col_k``), so every query leans towards those keys.
    Near slashes (offsets 0 .. near_offsets-1): a smooth positional code
    R[p] made of D/2 sinusoid pairs with frequencies spread over
    [0, pi / (2*near_offsets)] is added to queries and keys (``beta``), so a
    query leans towards keys at small offsets behind it.
    Far slashes: ``n_far_offsets`` random offsets o in [near_offsets, S/2); a
    sharp code P[p] with entries N(0,1)/sqrt(D) is added to the queries
    (Q[i] += alpha*P[i]) and to the keys (K[j] += alpha * sum_o P[j+o]).
    """
    rng = np.random.default_rng(seed)
    G = H_q // H_kv
    q = _normal_bits(rng, (B, S, H_q, D), True)
    k = _normal_bits(rng, (B, S, H_kv, D), True)
    v = _normal_bits(rng, (B, S, H_kv, D), True)
    cols = np.sort(rng.choice(S, size=min(n_columns, S), replace=False)).astype(np.int64)
    far_hi = max(near_offsets + 1, S // 2)
    n_far = min(n_far_offsets, max(0, far_hi - near_offsets))
    far = (np.sort(rng.choice(np.arange(near_offsets, far_hi), size=n_far, replace=False))
           if n_far else np.zeros(0, np.int64)).astype(np.int64)
    offsets = np.unique(np.concatenate([np.arange(min(near_offsets, S)), far])).astype(np.int64)
    e = rng.standard_normal((H_kv, D)).astype(np.float32)
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    # smooth code: cos/sin pairs, frequencies in [0, pi / (2 * near_offsets)]
    freq = rng.uniform(0.0, np.pi / (2 * near_offsets), size=D // 2)
    phase = rng.uniform(0.0, 2 * np.pi, size=D // 2)
    ang = np.arange(S)[:, None] * freq[None, :] + phase[None, :]
    R = (np.concatenate([np.cos(ang), np.sin(ang)], axis=1) / np.sqrt(D // 2)).astype(np.float32)
    span = S + (int(far.max()) + 1 if len(far) else 0)
    P = rng.standard_normal((span, D), dtype=np.float32) / np.float32(np.sqrt(D))
    Psum = np.zeros((S, D), np.float32)
    for o in far:
        Psum += P[o:o + S]
    for b in range(B):
        for h in range(H_q):
            qf = _as_f32(q[b, :, h, :], True)
            qf += beta * R + alpha * P[:S] + col_q * e[h // G]
            q[b, :, h, :] = _store(qf, True)
        for g in range(H_kv):
            kf = _as_f32(k[b, :, g, :], True)
            kf += beta * R + alpha * Psum
            kf[cols] += col_k * e[g]
            k[b, :, g, :] = _store(kf, True)
    return PrefillCase(name, B, S, H_q, H_kv, D, last_q, n_vertical, n_slash, q, k, v,
                       cols, offsets)


def prefill_128k() -> PrefillCase:
    """S=131072, 32 query heads over 8 KV heads, d=128, bf16, seed 4, top 1000 / 6096."""
    return prefill_case("prefill_vs_S131072", S=131072, H_q=32, H_kv=8, D=128, seed=4)
