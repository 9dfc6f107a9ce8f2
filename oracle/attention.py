"""fp64 CPU oracle: bf16 forward attention by its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by tests, the smoke
check and the CPU-baseline leg of the benchmark, never by the product.

Sources (web pages about MoonMath AI's bf16 forward-attention kernel):
  [DK] snilld.dk, "Open source attention-kernel i HIP slaar AITER v3 paa MI300X -
       hurtigere bf16-attention uden assembly".
         "Hvad er udgivet": BSHD and BHSD inputs without transpose, head_dim 128,
           arbitrary sequence lengths, cross-attention.
         "Hvordan kernen arbejder": the kernel computes softmax(QK^T/sqrt(d))*V and
           returns bf16.
         "Numerik samlet eet sted": bf16 output rounded per mode (the modes are
           named in the opening paragraph: one speedup per rounding mode); finite
           outputs within 1 bf16 ULP; NaN/Inf handled bit-identically;
           deterministic.
  [KO] tilnote.io note on the MoonMath HIP attention kernel for MI300X, section on
       the performance figures: the three modes are RTNE, RTNA and RTZ.

Readings where the pages are silent (each is listed in the design notes):
  * scale: any finite fp32; the pages' 1/sqrt(d) is the default. The oracle
    multiplies by (double)(float)scale so both sides use the same constant.
  * max is NaN-propagating; exp(s - m) is evaluated literally in IEEE fp64, so a
    +Inf logit gives a NaN row and a -Inf logit a zero weight (the safe-softmax
    reading, not a limit).
  * RTNE = nearest, ties to even; RTNA = nearest, ties away from zero; RTZ =
    toward zero. Rounded once, from the fp64 value. bf16 subnormals are kept.
    Overflow: RTNE/RTNA -> +-Inf, RTZ -> +-max finite.
  * every NaN output is written as the one pattern 0x7FC0.
  * causal (a follow-on step the pages name as missing): key j is visible to
    query i iff j <= i + (Sk - Sq), the bottom-right alignment that makes the last
    query see every key; hidden keys take no part (logit -Inf, and left out of the
    product with V), so a row that sees no key is NaN.
  * grouped-query attention (also named as missing): Hq query heads share Hkv
    key/value heads, query head h reads K/V head h // (Hq // Hkv).
  * variable-length batches (also named as missing, as cu_seqlens batching):
    sequences are packed token after token, Q as (total_q, Hq, d) and K, V as
    (total_k, Hkv, d); sequence b owns query rows cu_q[b]..cu_q[b+1]-1 and keys
    cu_k[b]..cu_k[b+1]-1 and attends only within itself. The causal alignment is
    per sequence. A sequence with queries but no keys gives NaN rows (the same
    reading as a row that sees no key).
"""
from __future__ import annotations

import numpy as np

MODES = ("rtne", "rtna", "rtz")

_ROW_BLOCK = 512


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16 / int16) -> float64 values (exact: bf16 is the top
    half of an IEEE binary32)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_bhsd(x: np.ndarray, layout: str) -> np.ndarray:
    """View a BSHD (batch, seq, head, dim) array as BHSD (batch, head, seq, dim).
    [DK] "Hvad er udgivet": both layouts describe the same tensor."""
    if layout == "bhsd":
        return x
    if layout == "bshd":
        return np.swapaxes(x, 1, 2)
    raise ValueError(f"unknown layout {layout!r}")


def _ieee_matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a @ b in fp64. BLAS when every operand is finite; otherwise an explicit
    sum of products, so that 0*Inf = NaN and NaN*0 = NaN hold exactly as IEEE
    says (a BLAS may skip zero operands)."""
    if np.isfinite(a).all() and np.isfinite(b).all():
        return a @ b
    return np.einsum("ik,kj->ij", a, b, optimize=False)


def attention_rows_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                        rows=None, causal: bool = False) -> np.ndarray:
    """O rows of one head, in fp64.

    q: (Sq, d), k: (Sk, d), v: (Sk, d), float64. rows: indices into Sq (default all).
    For each query row i ([DK] "Hvordan kernen arbejder", softmax(QK^T/sqrt(d))V):
      s_ij = scale * sum_c q_ic k_jc
      m_i  = max_j s_ij            (NaN if any s_ij is NaN)
      p_ij = exp(s_ij - m_i)
      l_i  = sum_j p_ij
      O_ic = (sum_j p_ij v_jc) / l_i
    The matrix products are library primitives; nothing is blocked or fused across
    the key axis. With causal, key j is hidden from row i when j > i + (Sk - Sq):
    s_ij = -Inf (so p_ij = 0), and the hidden keys take no part in the product
    either, so a non-finite value of V at a key a row does not see cannot reach
    that row (0 * NaN would).
    """
    scale_d = float(np.float32(scale))
    Sq_all, Sk = q.shape[0], k.shape[0]
    idx = np.arange(Sq_all) if rows is None else np.asarray(rows)
    q = q[idx]
    s = _ieee_matmul(q, k.T) * scale_d
    if causal:
        visible = np.clip(idx + (Sk - Sq_all) + 1, 0, Sk)  # keys 0 .. visible-1
        s = np.where(np.arange(Sk)[None, :] >= visible[:, None], -np.inf, s)
    with np.errstate(invalid="ignore", over="ignore"):
        m = np.max(s, axis=1, keepdims=True)  # np.max propagates NaN
        p = np.exp(s - m)
        l = np.sum(p, axis=1, keepdims=True)
        if causal and not np.isfinite(v).all():
            # Row by row over the visible keys only (a row that sees none is NaN).
            num = np.full((idx.size, v.shape[1]), np.nan)
            for r in range(idx.size):
                if visible[r] > 0:
                    num[r] = _ieee_matmul(p[r:r + 1, :visible[r]], v[:visible[r]])[0]
            o = num / l
        else:
            o = _ieee_matmul(p, v) / l
    return o


def attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   layout: str = "bhsd", causal: bool = False) -> np.ndarray:
    """Full attention for (B, H, S, d) or (B, S, H, d) float64 arrays.

    Returns O in the input layout (the pages' kernel reads either layout without a
    transpose; the output keeps the layout of the inputs). Rows are independent,
    so they are processed in groups of rows to bound memory. K and V may have
    fewer heads than Q (grouped-query attention, Hq a multiple of Hkv).
    """
    qb, kb, vb = to_bhsd(q, layout), to_bhsd(k, layout), to_bhsd(v, layout)
    B, H, Sq, d = qb.shape
    Hkv = kb.shape[1]
    if H % Hkv:
        raise ValueError("query heads must be a multiple of key/value heads")
    group = H // Hkv
    out = np.empty((B, H, Sq, d), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            kh, vh = kb[b, h // group], vb[b, h // group]
            for r0 in range(0, Sq, _ROW_BLOCK):
                rows = np.arange(r0, min(Sq, r0 + _ROW_BLOCK))
                out[b, h, rows] = attention_rows_fp64(qb[b, h], kh, vh, scale, rows, causal)
    if layout == "bshd":
        out = np.ascontiguousarray(np.swapaxes(out, 1, 2))
    return out


def round_bf16(x, mode: str) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (uint16) under one mode.

    bf16 has 8 significant bits and the binary32 exponent range. A finite nonzero
    |x| = f * 2**e with f in [0.5, 1) lies on the grid of spacing 2**(e-8) (normal
    range) or 2**-133 (subnormal range, |x| < 2**-126). The value is scaled onto
    that grid, split into integer and fraction exactly (both are exact in fp64),
    and the integer is bumped per the mode:
      rtne: fraction > 1/2, or = 1/2 with an odd integer
      rtna: fraction >= 1/2
      rtz : never
    A result of 2**128 or more is an overflow: Inf for rtne/rtna, max finite
    (0x7F7F) for rtz. NaN -> 0x7FC0. Signs (including -0) are kept.
    [DK] "Numerik samlet eet sted"; [KO] performance section (mode names).
    """
    if mode not in MODES:
        raise ValueError(f"unknown rounding mode {mode!r}")
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.zeros(flat.shape, dtype=np.uint32)
    neg = np.signbit(flat)
    a = np.abs(flat)
    nan = np.isnan(flat)
    inf = np.isinf(flat)
    fin = ~(nan | inf) & (a > 0)

    af = a[fin]
    _, e = np.frexp(af)
    qexp = np.maximum(e - 8, -133)
    r = np.ldexp(af, -qexp)
    n = np.floor(r)
    frac = r - n
    if mode == "rtne":
        up = (frac > 0.5) | ((frac == 0.5) & (np.fmod(n, 2.0) == 1.0))
    elif mode == "rtna":
        up = frac >= 0.5
    else:
        up = np.zeros(af.shape, dtype=bool)
    n = n + up
    with np.errstate(over="ignore"):
        val = np.ldexp(n, qexp)
    over = val >= 2.0 ** 128
    val32 = np.where(over, 0.0, val).astype(np.float32)
    bits = (val32.view(np.uint32) >> np.uint32(16)).astype(np.uint32)
    bits = np.where(over, np.uint32(0x7F7F if mode == "rtz" else 0x7F80), bits)
    out[fin] = bits
    out[inf] = 0x7F80
    out = np.where(neg, out | np.uint32(0x8000), out)
    out[nan] = 0x7FC0
    return out.astype(np.uint16).reshape(x.shape)


def nonfinite_bits(bits) -> np.ndarray:
    """True where a bf16 pattern is NaN or +-Inf."""
    b = np.asarray(bits).astype(np.uint16)
    return (b & np.uint16(0x7F80)) == np.uint16(0x7F80)


def ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Distance in bf16 ULPs between two bit patterns of finite values.

    Patterns map to an ordered integer line (negatives mirrored, +0 and -0 both 0);
    the distance is the difference on that line. Non-finite patterns are compared
    bit for bit elsewhere, not by this function.
    """
    def ordinal(x):
        x = np.asarray(x).astype(np.uint16).astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)

    return np.abs(ordinal(a_bits) - ordinal(b_bits))


def attention_varlen_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens_q,
                          cu_seqlens_k, scale: float, causal: bool = False) -> np.ndarray:
    """Attention over a packed batch of variable-length sequences, in fp64.

    The pages list variable-length ("varlen") batching among the features the
    kernel lacks ([DK] "Hvad er udgivet" and "Autoregressiv serving, de praktiske
    hager": production servers mix sequence lengths in one batch).

    q: (total_q, Hq, d); k, v: (total_k, Hkv, d); cu_seqlens_q / cu_seqlens_k: B+1
    non-decreasing offsets starting at 0 and ending at total_q / total_k. Each
    sequence is one (1, S, H, d) problem for attention_fp64; the result has q's
    shape. Rows of a sequence with no keys are NaN.
    """
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0:
        raise ValueError("cu_seqlens must have B+1 entries starting at 0")
    if any(b < a for a, b in zip(cq, cq[1:])) or any(b < a for a, b in zip(ck, ck[1:])):
        raise ValueError("cu_seqlens must be non-decreasing")
    if cq[-1] != q.shape[0] or ck[-1] != k.shape[0]:
        raise ValueError("cu_seqlens must end at the packed lengths")
    out = np.empty(q.shape, dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        if k1 == k0:
            out[q0:q1] = np.nan
            continue
        out[q0:q1] = attention_fp64(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], scale,
                                    layout="bshd", causal=causal)[0]
    return out
