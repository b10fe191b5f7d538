"""CPU oracle for the MoE layer hot path.  TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct restatement of what the layer computes, in
float64 with bfloat16 rounding applied only at the declared storage points.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it; the product path never does, and this module shares
no code with the CUDA path.

Source of the method: "Enabling trillion-parameter models on AWS EFA"
(Licker, Hu, Zaytsev, Chen; 2025).  The page fixes:
  * section "Introduction": an MoE layer replaces a dense layer with a set of
    experts plus a small linear routing layer that picks the experts a token is
    multiplied with; dispatch splits the tokens by expert, and combine, its
    dual, gathers the processed tokens back and takes their weighted average;
  * section "Send and receive buffers": T tokens, each routed to R of E experts;
  * section "Dispatch and combine": per-expert token counts, then a cumulative
    sum of the counts gives the offsets that pack the tokens of each expert
    contiguously; the receiver shuffles tokens into the tensor the grouped
    GEMM consumes, and combine accumulates the weighted tokens at the receiver;
  * section "MoE all-to-all over EFA": dispatch -> grouped GEMMs multiply the
    tokens by the expert weights -> combine returns them and averages.
Readings where the page is silent (all listed in the design notes):
  * router: logits = x @ W_g + bias in fp32; experts ordered by (logit desc,
    index asc); the first R are chosen, in that order; the gate weights are the
    softmax of the chosen logits (renormalised top-R softmax), so they sum to 1;
  * within an expert, rows are ordered by ascending token index;
  * expert FFN: SwiGLU, h = silu(x W1^T) * (x W3^T), o = h W2^T;
  * bf16 round-to-nearest-even at h, o, y (forward) and at do, da, db,
    dx_perm, dx (backward); a and b are kept for the backward as bf16;
  * loss L = sum(y * g); no auxiliary loss; the router bias is a constant;
  * shared expert (section "Introduction": the GPU multiplies the shared
    expert while dispatch is in flight): a SwiGLU FFN that every token passes
    through, its output s = bf16(h_s Ws2^T) added to the routed experts'
    weighted sum with weight 1, y = bf16(s + sum_r w_r o_r); its backward
    takes dy as the output gradient.

Parity pins for every function live in tests/test_oracle.py.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
# ----------------------------------------------------------------------------
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_QUANTUM_EXP = -133      # spacing of bf16 subnormals: 2^(-126-7)


def bf16_round(v, enabled: bool = True):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    Written from the IEEE 754 definition: a finite nonzero value |v| in
    [2^k, 2^(k+1)) keeps 8 significant bits, so the representable spacing there
    is 2^(k-7) (never finer than the subnormal spacing 2^-133).  |v|/spacing is
    rounded to the nearest integer with ties to even (np.rint) and scaled back;
    both scalings are exact in float64.  Results above the largest finite bf16
    value overflow to infinity.  With ``enabled=False`` the values pass through
    unchanged (used to check gradients by finite differences).
    """
    v = np.asarray(v, dtype=np.float64)
    if not enabled:
        return v.copy()
    out = v.copy()
    fin = np.isfinite(v) & (v != 0.0)
    a = np.abs(v[fin])
    _, e = np.frexp(a)                       # a = m * 2^e, 0.5 <= m < 1
    q = np.ldexp(1.0, np.maximum(e - 1 - 7, _BF16_MIN_QUANTUM_EXP))
    r = np.rint(a / q) * q
    r[r > BF16_MAX] = np.inf
    out[fin] = np.copysign(r, v[fin])
    return out


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def values(a):
    """bf16 bit patterns (uint16) -> float64 values; other arrays -> float64 as is."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f64(a)
    return a.astype(np.float64)


def f64_to_bf16_bits(v):
    """float64 values that are already bf16-representable -> uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# Routing: a small linear layer scores the experts for each token and the best
# ones are chosen (section "Introduction").
# ----------------------------------------------------------------------------
def gate_logits(x, w_gate, bias=None, rounding=True):
    """logits[t,e] = sum_k x[t,k] * W_g[k,e] + bias[e]; float64 sums, stored fp32.

    With ``rounding=False`` the float64 sums are returned unrounded.
    """
    x = values(x)
    l = x @ np.asarray(w_gate, dtype=np.float64)
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l.astype(np.float32) if rounding else l


def route_topk(logits, R):
    """Top-R expert choice and gate weights for each token.

    Experts are ordered by (fp32 logit descending, expert index ascending); the
    first R are taken, in that order (idx[t, 0] is the best expert).  The gate
    weights are the softmax of the chosen logits,
        w_r = exp(l_{i_r} - l_{i_0}) / sum_s exp(l_{i_s} - l_{i_0}),
    so they are positive and sum to 1 (combine is a weighted average).
    Returns idx int32 [T,R] and w [T,R] (computed in float64; stored float32
    when the logits are float32, kept float64 when they are float64).
    """
    l = np.asarray(logits)
    assert l.dtype in (np.float32, np.float64)
    T, E = l.shape
    assert 1 <= R <= E
    key_index = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((key_index, -l), axis=-1)     # primary: -logit, then index
    idx = order[:, :R].astype(np.int32)
    sel = np.take_along_axis(l, idx, axis=1).astype(np.float64)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w.astype(l.dtype)


# ----------------------------------------------------------------------------
# Dispatch (section "Dispatch and combine": per-expert counts, cumulative sum
# for contiguous offsets, shuffle into the grouped-GEMM input).
# ----------------------------------------------------------------------------
def dispatch_plan(idx, E):
    """counts[E], offsets[E+1], row_slot[N], slot_row[N] for N = T*R slots.

    A slot is s = t*R + r.  counts[e] = #{s : idx_s = e}; offsets is their
    exclusive cumulative sum (offsets[E] = N).  Within expert e the rows
    offsets[e] .. offsets[e+1]-1 hold its slots in ascending token order (a
    token names an expert at most once, so ascending slot order is the same).
    row_slot[row] = slot; slot_row[slot] = row (mutually inverse).
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < E)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    row_slot = np.argsort(flat, kind="stable").astype(np.int32)
    slot_row = np.empty_like(row_slot)
    slot_row[row_slot] = np.arange(flat.size, dtype=np.int32)
    return counts, offsets, row_slot, slot_row


def permute_rows(x, row_slot, R):
    """x_perm[row] = x[token of row_slot[row]] (a copy; bit patterns stay bit patterns)."""
    return np.asarray(x)[np.asarray(row_slot) // R].copy()


# ----------------------------------------------------------------------------
# Grouped SwiGLU expert FFN: after dispatch, grouped GEMMs apply each expert's
# weights to the tokens routed to it (section "MoE all-to-all over EFA").
# ----------------------------------------------------------------------------
def silu(a):
    return a / (1.0 + np.exp(-a))


def expert_ffn(x_perm, offsets, W1, W3, W2, rounding=True, row_scale=None):
    """Per expert e over rows offsets[e]..offsets[e+1]-1 of x_perm:

        a = x W1[e]^T, b = x W3[e]^T      (float64)
        h = bf16(silu(a) * b)
        o = bf16(s * (h W2[e]^T))         s = row_scale[row] (1 when None)

    ``row_scale`` weights each output row before its rounding (e.g. by the
    row's gate weight, so that an unweighted combine sums weighted rows).

    W1, W3: [E, f, d]; W2: [E, d, f] (bf16 bit patterns or float64 values; an
    expert's weights are decoded only when its rows are processed).
    Returns a, b (float64), h, o (float64 holding bf16 values).
    """
    E = len(offsets) - 1
    N = int(offsets[-1])
    f = W1.shape[1]
    d = W1.shape[2]
    a = np.zeros((N, f))
    b = np.zeros((N, f))
    h = np.zeros((N, f))
    o = np.zeros((N, d))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        xe = values(x_perm[r0:r1])
        ae = xe @ values(W1[e]).T
        be = xe @ values(W3[e]).T
        he = bf16_round(silu(ae) * be, rounding)
        pe = he @ values(W2[e]).T
        if row_scale is not None:
            pe = np.asarray(row_scale, dtype=np.float64)[r0:r1, None] * pe
        oe = bf16_round(pe, rounding)
        a[r0:r1], b[r0:r1], h[r0:r1], o[r0:r1] = ae, be, he, oe
    return a, b, h, o


# ----------------------------------------------------------------------------
# Combine: each token's expert outputs come back to it and are averaged with
# the gate weights (section "Introduction"); the sum is taken at the token's
# side (section "Dispatch and combine").
# ----------------------------------------------------------------------------
def combine(o, slot_row, w, T, R, rounding=True, add=None):
    """y[t] = bf16( add[t] + sum_{r=0..R-1} w[t,r] * o[slot_row[t*R+r]] ), summed in r order.

    ``o`` holds float64 values; ``w`` None means unweighted (all ones); ``add``
    (the shared expert's output rows, [T, d]) None means zero.
    """
    o = np.asarray(o, dtype=np.float64)
    y = np.zeros((T, o.shape[1])) if add is None else np.array(add, dtype=np.float64)
    sr = np.asarray(slot_row).reshape(T, R)
    for r in range(R):
        wr = 1.0 if w is None else np.asarray(w, dtype=np.float64)[:, r:r + 1]
        y = y + wr * o[sr[:, r]]
    return bf16_round(y, rounding)


# ----------------------------------------------------------------------------
# Block-scaled fp8 dispatch ("Enabling trillion-parameter models on AWS EFA",
# section "Evaluation": tokens are dispatched in block-scaled fp8 and combined
# in bf16).  Reading: E4M3 codes (the OCP 8-bit E4M3 format without
# infinities), one fp32 scale per token and 128 consecutive hidden channels,
# scale = amax / 448 so the block's largest magnitude maps to the largest
# finite code; codes are rounded to nearest even from the fp32 quotient
# x / scale and saturate at +-448.
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0
FP8_BLOCK = 128


def e4m3_decode(codes):
    """E4M3 bit patterns (uint8) -> float64: 1 sign, 4 exponent bits (bias 7),
    3 fraction bits; exponent 0 is subnormal (fraction * 2^-9); exponent 15 with
    fraction 7 is NaN; there are no infinities."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    ex = (b >> 3) & 0xF
    fr = b & 0x7
    mag = np.where(ex == 0, fr * 2.0 ** -9, (1.0 + fr / 8.0) * np.ldexp(1.0, ex - 7))
    mag = np.where((ex == 15) & (fr == 7), np.nan, mag)
    return sign * mag


def e4m3_round(v):
    """Nearest E4M3 value, ties to even, magnitudes above 448 saturate to 448.

    A value |v| in [2^k, 2^(k+1)) with k >= -6 keeps 4 significant bits
    (spacing 2^(k-3)); below 2^-6 the spacing is the subnormal step 2^-9.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)                                  # a = m 2^e, 0.5 <= m < 1
    q = np.ldexp(1.0, np.maximum(e - 1 - 3, -9))
    r = np.rint(a / q) * q
    r = np.where(a == 0, 0.0, np.minimum(r, E4M3_MAX))
    return np.copysign(r, v)


def e4m3_encode(vals):
    """E4M3-representable float64 values -> their uint8 codes (-0 -> 0x80), by
    lookup in the sorted table of the 254 finite code values."""
    table = e4m3_decode(np.arange(256, dtype=np.uint8))
    codes = np.array([c for c in range(256) if np.isfinite(table[c]) and c != 0x80], np.uint8)
    order = np.argsort(table[codes], kind="stable")
    tv, codes = table[codes][order], codes[order]
    v = np.asarray(vals, dtype=np.float64).ravel()
    pos = np.clip(np.searchsorted(tv, v), 0, len(tv) - 1)
    assert np.array_equal(tv[pos], v), "value not representable in E4M3"
    out = codes[pos]
    out[(v == 0) & np.signbit(v)] = 0x80
    return out.reshape(np.shape(vals))


def quantize_fp8_blocks(x):
    """Per token and 128-channel block: scale = fp32(amax / 448), codes =
    e4m3(fp32(x / scale)).  x: bf16 bits or values [T, d] with d % 128 == 0.
    Returns codes uint8 [T, d] and scales float32 [T, d/128]; an all-zero block
    has scale 0 and zero codes."""
    xv = values(x).astype(np.float32)
    T, d = xv.shape
    assert d % FP8_BLOCK == 0
    blocks = xv.reshape(T, d // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2)
    scales = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scales > 0, scales, np.float32(1.0))
    quot = (blocks / safe[:, :, None]).astype(np.float32)       # fp32 quotient
    vals = e4m3_round(quot.astype(np.float64))
    vals = np.where(scales[:, :, None] > 0, vals, 0.0)
    return e4m3_encode(vals).reshape(T, d), scales


def dequantize_fp8_blocks(codes, scales):
    """codes [N, d] uint8, scales [N, d/128] -> float64 values code * scale."""
    c = e4m3_decode(codes)
    N, d = c.shape
    return (c.reshape(N, d // FP8_BLOCK, FP8_BLOCK) * np.asarray(scales, np.float64)[:, :, None]
            ).reshape(N, d)


# ----------------------------------------------------------------------------
# Microscaled fp8 for the expert GEMMs ("Enabling trillion-parameter models on
# AWS EFA", section "Evaluation": the tokens travel as block-scaled fp8).
# Reading for GEMMs that consume fp8 directly (the tensor cores' block-scaled
# fp8 multiply takes one power-of-two scale per 32 consecutive elements along
# the contraction): E4M3 codes, one UE8M0 scale (a power of two, stored as its
# exponent + 127) per 32 consecutive elements of a row along K.  The scale of a
# block is the smallest power of two 2^k with 448 * 2^k >= amax (so no code
# saturates), k clamped to [-127, 127]; codes are the E4M3 values nearest to
# x / 2^k, ties to even.  An all-zero block gets k = -127 (code 0) and zero
# codes.  Weights are quantised the same way along their K (d for W1 and W3,
# f for W2); the expert FFN quantises h = silu(a) * b the same way along f
# before the down projection.
# ----------------------------------------------------------------------------
MX_BLOCK = 32
MX_BIAS = 127


def mx_scale_exponents(amax):
    """Per block: the smallest integer k with 448 * 2^k >= amax, clamped to
    [-127, 127] (k = -127 for amax = 0).  Exact: with amax = m * 2^e,
    0.5 <= m < 1 and 448 = 0.875 * 2^9, k = e - 9 when m <= 0.875, else e - 8."""
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)
    k = np.where(m <= 0.875, e - 9, e - 8)
    k = np.where(a == 0, -MX_BIAS, k)
    return np.clip(k, -MX_BIAS, MX_BIAS).astype(np.int64)


def quantize_mx(x):
    """x: [rows, K] (bf16 bits or values), K % 32 == 0.  Returns E4M3 codes
    uint8 [rows, K] and scale codes uint8 [rows, K/32] (k + 127)."""
    xv = values(x)
    rows, K = xv.shape
    assert K % MX_BLOCK == 0
    blocks = xv.reshape(rows, K // MX_BLOCK, MX_BLOCK)
    k = mx_scale_exponents(np.abs(blocks).max(axis=2))
    q = e4m3_round(blocks / np.ldexp(1.0, k)[:, :, None])      # exact division by 2^k
    return e4m3_encode(q).reshape(rows, K), (k + MX_BIAS).astype(np.uint8)


def dequantize_mx(codes, scales):
    """codes uint8 [rows, K], scale codes uint8 [rows, K/32] -> float64 values."""
    c = e4m3_decode(codes)
    rows, K = c.shape
    k = np.asarray(scales, dtype=np.int64)[:, : K // MX_BLOCK] - MX_BIAS
    return (c.reshape(rows, K // MX_BLOCK, MX_BLOCK) * np.ldexp(1.0, k)[:, :, None]).reshape(rows, K)


def expert_ffn_mx(xq, xs, offsets, W1q, W1s, W3q, W3s, W2q, W2s, quantize_h=True, row_scale=None):
    """The expert FFN on microscaled fp8 operands.  Per expert e over its rows:

        x = dequant(xq, xs);  w1, w3, w2 = dequant(W*q[e], W*s[e])
        a = x w1^T, b = x w3^T,  hv = silu(a) * b          (float64)
        hq, hs = quantize_mx(hv) along f;  h = dequant(hq, hs)   (hv itself
                                                    when quantize_h is False)
        o = bf16(s * (h w2^T))                              s = row_scale[row] or 1

    W1q, W3q: uint8 [E, f, d] with scales [E, f, d/32]; W2q: uint8 [E, d, f]
    with scales [E, d, f/32].  Returns a, b, hv, hq, hs, h, o.
    """
    E = len(offsets) - 1
    N = int(offsets[-1])
    f, d = W1q.shape[1], W1q.shape[2]
    a = np.zeros((N, f))
    b = np.zeros((N, f))
    hv = np.zeros((N, f))
    h = np.zeros((N, f))
    hq = np.zeros((N, f), dtype=np.uint8)
    hs = np.zeros((N, f // MX_BLOCK), dtype=np.uint8)
    o = np.zeros((N, d))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        x = dequantize_mx(xq[r0:r1], xs[r0:r1])
        ae = x @ dequantize_mx(W1q[e], W1s[e]).T
        be = x @ dequantize_mx(W3q[e], W3s[e]).T
        ve = silu(ae) * be
        if quantize_h:
            qe, se = quantize_mx(ve)
            he = dequantize_mx(qe, se)
            hq[r0:r1], hs[r0:r1] = qe, se
        else:
            he = ve
        pe = he @ dequantize_mx(W2q[e], W2s[e]).T
        if row_scale is not None:
            pe = np.asarray(row_scale, dtype=np.float64)[r0:r1, None] * pe
        a[r0:r1], b[r0:r1], hv[r0:r1], h[r0:r1] = ae, be, ve, he
        o[r0:r1] = bf16_round(pe)
    return a, b, hv, hq, hs, h, o


# ----------------------------------------------------------------------------
# Whole layer.
# ----------------------------------------------------------------------------
def shared_expert_fwd(x, Ws1, Ws3, Ws2, rounding=True):
    """The shared expert: the expert FFN with one expert holding every token,
    rows in token order.  Returns (a, b, h, s) as ``expert_ffn`` does."""
    T = np.asarray(x).shape[0]
    offsets = np.array([0, T], dtype=np.int64)
    return expert_ffn(x, offsets, np.asarray(Ws1)[None], np.asarray(Ws3)[None],
                      np.asarray(Ws2)[None], rounding)


def layer_fwd(x, w_gate, bias, W1, W3, W2, R, rounding=True,
              forced_idx=None, forced_w=None, shared=None):
    """Forward pass of the MoE layer: route -> dispatch -> expert FFN -> combine.

    ``forced_idx``/``forced_w`` replace the router's choice (used to compare the
    later stages with a GPU run whose routing is fixed).  ``shared`` = (Ws1,
    Ws3, Ws2) adds a shared expert.  Returns a dict of all intermediates; bf16
    tensors are float64 arrays holding bf16 values.
    """
    x = np.asarray(x)
    T = x.shape[0]
    E = W1.shape[0]
    logits = gate_logits(x, w_gate, bias, rounding)
    if forced_idx is None:
        idx, w = route_topk(logits, R)
    else:
        idx, w = np.asarray(forced_idx, np.int32), np.asarray(forced_w)
    counts, offsets, row_slot, slot_row = dispatch_plan(idx, E)
    x_perm = permute_rows(x, row_slot, R)
    a, b, h, o = expert_ffn(x_perm, offsets, W1, W3, W2, rounding)
    out = {}
    s_out = None
    if shared is not None:
        sa, sb, sh, s_out = shared_expert_fwd(x, *shared, rounding=rounding)
        out.update(sa=sa, sb=sb, sh=sh, s=s_out)
    y = combine(o, slot_row, w, T, R, rounding, add=s_out)
    out.update(logits=logits, idx=idx, w=w, counts=counts, offsets=offsets, row_slot=row_slot,
               slot_row=slot_row, x_perm=x_perm, a=a, b=b, h=h, o=o, y=y)
    return out


def expert_bwd(x_rows, a, b, h, do, W1e, W3e, W2e, rounding=True):
    """Backward of one expert's SwiGLU FFN over its rows (float64).

    a, b: the forward pre-activations (kept as bf16 for the backward); h: the
    forward hidden rows; do: the rows' output gradients (bf16 values).
        dh      = do W2e
        da      = bf16(dh * b_s * silu'(a_s)),  db = bf16(dh * silu(a_s)),
                  a_s = bf16(a), b_s = bf16(b), silu'(a) = s(a)(1 + a(1 - s(a)))
        dx_perm = bf16(da W1e + db W3e)
        dW2e = do^T h,  dW1e = da^T x,  dW3e = db^T x
    """
    x_rows = values(x_rows)
    w1, w3, w2 = values(W1e), values(W3e), values(W2e)
    a_s = bf16_round(a, rounding)
    b_s = bf16_round(b, rounding)
    dh = do @ w2
    sg = 1.0 / (1.0 + np.exp(-a_s))
    dsilu = sg * (1.0 + a_s * (1.0 - sg))
    da = bf16_round(dh * b_s * dsilu, rounding)
    db = bf16_round(dh * a_s * sg, rounding)
    return dict(da=da, db=db, dx_perm=bf16_round(da @ w1 + db @ w3, rounding),
                dW2=do.T @ h, dW1=da.T @ x_rows, dW3=db.T @ x_rows)


def layer_bwd(fwd, x, w_gate, W1, W3, W2, dy, R, rounding=True, shared=None):
    """Backward pass for L = sum(y * g) with dy = g (bf16 bits or float64 values).

    Per token t and slot r (row = slot_row[t*R+r], expert e = idx[t,r]):
        dw[t,r]   = <dy_t, o_row>
        do_row    = bf16(w[t,r] * dy_t)
    Per expert e (rows of e), with a_s = bf16(a), b_s = bf16(b) as saved:
        dh        = do W2[e]                                  (no rounding)
        da        = bf16(dh * b_s * silu'(a_s)),  silu'(a) = s(a) (1 + a (1 - s(a)))
        db        = bf16(dh * silu(a_s))
        dx_perm   = bf16(da W1[e] + db W3[e])
        dW2[e]    = do^T h,  dW1[e] = da^T x_perm,  dW3[e] = db^T x_perm
    Router (softmax over the chosen logits; unchosen logits get no gradient):
        dlogits[t, idx[t,q]] = w_q (dw_q - sum_r w_r dw_r)
        dW_g      = x^T dlogits
        dx_t      = bf16( sum_r dx_perm[row(t,r)] + dlogits_t W_g^T [+ dxs_t] )
    Shared expert (``shared`` = (Ws1, Ws3, Ws2); its output gradient is dy):
        dxs, dWs1, dWs3, dWs2 as ``expert_bwd`` over all T rows with do = dy.
    Returns dict with dx, dW_gate, dW1, dW3, dW2 (float64) and intermediates.
    """
    x = values(x)
    dy = values(dy)
    T = x.shape[0]
    E = W1.shape[0]
    idx, w = fwd["idx"], fwd["w"].astype(np.float64)
    offsets, slot_row = fwd["offsets"], fwd["slot_row"]
    sr = np.asarray(slot_row).reshape(T, R)
    o = fwd["o"]
    N = o.shape[0]
    d = o.shape[1]
    f = fwd["h"].shape[1]

    dw = np.zeros((T, R))
    do = np.zeros((N, d))
    for r in range(R):
        rows = sr[:, r]
        dw[:, r] = np.sum(dy * o[rows], axis=1)
        do[rows] = bf16_round(w[:, r:r + 1] * dy, rounding)

    x_perm = values(fwd["x_perm"])
    dx_perm = np.zeros((N, d))
    da = np.zeros((N, f))
    db = np.zeros((N, f))
    dW1 = np.zeros((E, f, d))
    dW3 = np.zeros((E, f, d))
    dW2 = np.zeros((E, d, f))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        eb = expert_bwd(x_perm[r0:r1], fwd["a"][r0:r1], fwd["b"][r0:r1], fwd["h"][r0:r1],
                        do[r0:r1], W1[e], W3[e], W2[e], rounding)
        dx_perm[r0:r1], da[r0:r1], db[r0:r1] = eb["dx_perm"], eb["da"], eb["db"]
        dW1[e], dW3[e], dW2[e] = eb["dW1"], eb["dW3"], eb["dW2"]

    wdw = np.sum(w * dw, axis=1, keepdims=True)
    dsel = w * (dw - wdw)
    dlogits = np.zeros((T, E))
    np.put_along_axis(dlogits, np.asarray(idx, np.int64), dsel, axis=1)
    wg = np.asarray(w_gate, dtype=np.float64)
    dW_gate = x.T @ dlogits
    dx = np.zeros((T, d))
    for r in range(R):
        dx = dx + dx_perm[sr[:, r]]
    dx = dx + dlogits @ wg.T
    out = {}
    if shared is not None:
        sb_ = expert_bwd(x, fwd["sa"], fwd["sb"], fwd["sh"], dy, *shared, rounding=rounding)
        dx = dx + sb_["dx_perm"]
        out.update(dxs=sb_["dx_perm"], dWs1=sb_["dW1"], dWs3=sb_["dW3"], dWs2=sb_["dW2"],
                   das=sb_["da"], dbs=sb_["db"])
    dx = bf16_round(dx, rounding)
    out.update(dx=dx, dW_gate=dW_gate, dW1=dW1, dW3=dW3, dW2=dW2, dw=dw, do=do, da=da, db=db,
               dx_perm=dx_perm, dlogits=dlogits)
    return out


def loss(y, g):
    """L = sum(y * g) in float64."""
    return float(np.sum(np.asarray(y, np.float64) * np.asarray(g, np.float64)))
