"""fp64 CPU oracle of the Megatron-Core-style MoE expert layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference legs may import this module.  The CUDA
library never calls it, shares no code with it and it imports nothing from the
library.  It is deliberately plain and slow: numpy fp64, one step per function,
in the order the layer is defined.

Source: "Scalable Training of Mixture-of-Experts Models with Megatron Core"
(summary page).  What each step follows there:

* routing to a few experts per token: "Problem" section 1 (each input goes to
  the two or three best-suited experts, the rest idle);
* the router is kept in high precision: technical summary section 2.5
  (selective precision: router, embedding and optimizer state stay FP32/BF16);
* permutation of tokens into expert order with dynamic shapes, no host sync:
  technical summary section 1, compute-efficiency wall, and section 2.4
  (sync-free kernels: the GPU reads the shape information itself);
* grouped GEMM over all experts: technical summary section 2.4;
* routing weight applied before the activation computation so backward keeps
  no extra intermediate: technical summary section 2.2 (memory-efficient
  permutation);
* MXFP8 expert GEMMs on Blackwell: technical summary section 2.5;
* NVFP4 expert GEMMs, named beside MXFP8 in the same section (forward only;
  the format's own definition is the reading, see the NVFP4 section below).

The pages give no formula for any of these.  The readings taken where they are
silent (gate formulas, selection key, tie rule, SwiGLU layout, where the gate
multiplies, the MX scale rule, the NVFP4 tensor scale) are listed with the design notes of the
repository; each function below states the reading it implements.

Every function here is pinned by a test in tests/test_oracle_*.py against
something other than itself (brute force, closed forms, invariants, library
routines, finite differences).  Parity pinned for all functions.
"""
from __future__ import annotations

import numpy as np

SOFTMAX = "softmax"
SIGMOID = "sigmoid"


# ---------------------------------------------------------------------------
# Router (technical summary 2.5: router stays in high precision)
# ---------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """logits[t, e] = <x_t, Wr_e>, fp64.  x [T,H], Wr [E,H] -> [T,E]."""
    return np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T


def _shape(a):
    """Shape of an array, or of an object that only exposes ``shape`` and
    per-expert indexing (lets a test stream expert weights in one at a time)."""
    return a.shape if hasattr(a, "shape") else np.asarray(a).shape


def _sigmoid(v: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-v))


def selection_keys(logits: np.ndarray, score: str, bias=None) -> np.ndarray:
    """Key each expert is ranked by.

    softmax scoring: the logit itself (softmax is monotone, so ranking the raw
    logit ranks the probability, without creating ties by rounding).
    sigmoid scoring: sigmoid(logit) + bias_e; the bias changes only which
    experts are chosen, never the gate values.
    """
    logits = np.asarray(logits, np.float64)
    if score == SOFTMAX:
        return logits.copy()
    if score == SIGMOID:
        b = 0.0 if bias is None else np.asarray(bias, np.float64)[None, :]
        return _sigmoid(logits) + b
    raise ValueError(score)


def selection_keys_f32(logits_f32: np.ndarray, score: str, bias=None) -> np.ndarray:
    """The same keys, computed in float32 (the kernel's precision for this
    decision).  Used where an fp32 choice must be reproduced exactly."""
    l32 = np.asarray(logits_f32, np.float32)
    if score == SOFTMAX:
        return l32.copy()
    one = np.float32(1.0)
    s = one / (one + np.exp(-l32))
    if bias is not None:
        s = s + np.asarray(bias, np.float32)[None, :]
    return s.astype(np.float32)


def topk_select(keys: np.ndarray, k: int) -> np.ndarray:
    """For each token, the k experts with the largest key, ordered by key
    descending; equal keys go to the lower expert id first.  [T,E] -> [T,k] int32."""
    keys = np.asarray(keys)
    T, E = keys.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary.  Primary: key descending; secondary: id ascending.
    order = np.lexsort((ids, -keys), axis=-1)
    return order[:, :k].astype(np.int32)


def topk_gap(keys: np.ndarray, k: int) -> np.ndarray:
    """Per token, key_(k) - key_(k+1) (inf when k == E): how close the choice of
    the k-th expert was.  Tokens with a small gap may be routed differently by a
    computation that rounds differently."""
    keys = np.asarray(keys, np.float64)
    T, E = keys.shape
    if k >= E:
        return np.full(T, np.inf)
    srt = -np.sort(-keys, axis=-1)
    gap = srt[:, k - 1] - srt[:, k]
    # also the smallest gap among the chosen ones (order inside the top-k)
    if k > 1:
        inner = np.min(srt[:, :k - 1] - srt[:, 1:k], axis=-1)
        gap = np.minimum(gap, inner)
    return gap


def gates_from_logits(logits: np.ndarray, sel: np.ndarray, score: str) -> np.ndarray:
    """Gate weights of the chosen experts, normalised over the chosen set.

    softmax: g_i = exp(l_{S_i}) / sum_{j in S} exp(l_j)   (equal to a full softmax
             renormalised over S, so both wordings give one function);
    sigmoid: g_i = sig(l_{S_i}) / sum_{j in S} sig(l_j)  (no extra scale factor).
    """
    logits = np.asarray(logits, np.float64)
    l_sel = np.take_along_axis(logits, sel.astype(np.int64), axis=-1)
    if score == SOFTMAX:
        m = l_sel.max(axis=-1, keepdims=True)
        e = np.exp(l_sel - m)
        return e / e.sum(axis=-1, keepdims=True)
    if score == SIGMOID:
        s = _sigmoid(l_sel)
        return s / s.sum(axis=-1, keepdims=True)
    raise ValueError(score)


def route(logits: np.ndarray, k: int, score: str, bias=None):
    """Top-k routing of fp64 logits: returns (topk_idx [T,k] int32, gates [T,k] fp64)."""
    keys = selection_keys(logits, score, bias)
    sel = topk_select(keys, k)
    return sel, gates_from_logits(logits, sel, score)


# ---------------------------------------------------------------------------
# Permutation into expert-contiguous order (technical summary 1 and 2.4:
# dynamic shapes, sync-free; the shape information is counts and offsets)
# ---------------------------------------------------------------------------

def permutation_maps(topk_idx: np.ndarray, E: int, pad: int = 128) -> dict:
    """Expert-contiguous row layout of the T*k (token, slot) pairs.

    counts[e]   number of pairs routed to expert e
    offsets     exclusive scan of counts (compact layout), length E+1
    poffsets    exclusive scan of counts rounded up to ``pad`` rows, length E+1
    slot_row    [T,k]: padded row of pair (t,i) = poffsets[e] + rank, where rank is
                the number of earlier tokens t' < t routed to the same expert
                (a stable counting sort by expert)
    row_src     [poffsets[E]]: token of each padded row, -1 for padding rows
    row_slot    [poffsets[E]]: slot i of each padded row, -1 for padding rows
    """
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, np.int64)
    for t in range(T):
        for i in range(k):
            counts[idx[t, i]] += 1
    offsets = np.zeros(E + 1, np.int64)
    poffsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
        poffsets[e + 1] = poffsets[e] + ((counts[e] + pad - 1) // pad) * pad
    slot_row = np.zeros((T, k), np.int64)
    row_src = np.full(int(poffsets[E]), -1, np.int64)
    row_slot = np.full(int(poffsets[E]), -1, np.int64)
    seen = np.zeros(E, np.int64)
    for t in range(T):                  # ascending t: the order inside an expert
        for i in range(k):
            e = idx[t, i]
            r = poffsets[e] + seen[e]
            seen[e] += 1
            slot_row[t, i] = r
            row_src[r] = t
            row_slot[r] = i
    return {"counts": counts, "offsets": offsets, "poffsets": poffsets,
            "slot_row": slot_row, "row_src": row_src, "row_slot": row_slot}


def compact_rows(maps: dict) -> np.ndarray:
    """Compact position offsets[e] + rank of each pair, [T,k] (same rank as slot_row)."""
    pos = maps["slot_row"].copy()
    po, of = maps["poffsets"], maps["offsets"]
    E = len(po) - 1
    for e in range(E):
        m = (pos >= po[e]) & (pos < po[e + 1])
        pos[m] = pos[m] - po[e] + of[e]
    return pos


def permute(x: np.ndarray, maps: dict) -> np.ndarray:
    """x_perm[r] = x[row_src[r]], zero rows for padding."""
    x = np.asarray(x)
    src = maps["row_src"]
    out = np.zeros((len(src),) + x.shape[1:], np.float64)
    valid = src >= 0
    out[valid] = x[src[valid]]
    return out


def unpermute_sum(o_perm: np.ndarray, maps: dict, shared=None) -> np.ndarray:
    """y[t] = sum_i o_perm[slot_row[t,i]] (+ shared[t]); unweighted, because the
    gate has already been applied inside the expert (technical summary 2.2)."""
    slot_row = maps["slot_row"]
    y = np.asarray(o_perm, np.float64)[slot_row].sum(axis=1)
    if shared is not None:
        y = y + np.asarray(shared, np.float64)
    return y


# ---------------------------------------------------------------------------
# Expert MLP (SwiGLU).  W1_e = [W_gate; W_up] of shape [2F,H]; W2_e is [H,F].
# ---------------------------------------------------------------------------

def silu(v):
    return v * _sigmoid(v)


def silu_grad(v):
    s = _sigmoid(v)
    return s * (1.0 + v * (1.0 - s))


def swiglu_expert(x_rows: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """W2 ( silu(W_gate x) * (W_up x) ) for each row of x_rows."""
    w1 = np.asarray(w1, np.float64)
    F = w1.shape[0] // 2
    z = np.asarray(x_rows, np.float64) @ w1.T
    h = silu(z[:, :F]) * z[:, F:]
    return h @ np.asarray(w2, np.float64).T


# ---------------------------------------------------------------------------
# The layer
# ---------------------------------------------------------------------------

def moe_forward(x, w_router, w1, w2, k, score=SOFTMAX, bias=None,
                w1_shared=None, w2_shared=None, routing=None, expert_fn=None):
    """y_t = sum_i g_{t,i} * Expert_{S_t[i]}(x_t)  (+ SharedExpert(x_t)).

    ``routing`` = (topk_idx, gates) replaces the router (router replay, or the
    GPU's own routing when comparing the expert path alone).
    ``expert_fn(e, rows)`` replaces the SwiGLU expert (used by the identity pin).
    Returns a dict with y and the routing record.
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = _shape(w_router)[0] if w_router is not None else _shape(w1)[0]
    logits = None
    if routing is None:
        logits = router_logits(x, w_router)
        idx, gate = route(logits, k, score, bias)
    else:
        idx = np.asarray(routing[0], np.int64)
        gate = np.asarray(routing[1], np.float64)
    y = np.zeros_like(x)
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        rows = x[tok]
        out = expert_fn(e, rows) if expert_fn is not None else swiglu_expert(rows, w1[e], w2[e])
        np.add.at(y, tok, gate[tok, slot][:, None] * out)
    if w1_shared is not None:
        y += swiglu_expert(x, w1_shared, w2_shared)
    return {"y": y, "logits": logits, "topk_idx": idx.astype(np.int32), "gates": gate}


def router_backward(logits, sel, gates, dgate, score):
    """dlogits [T,E] from the gate gradient.  Only the chosen experts' logits
    receive gradient; the selection bias receives none.

    softmax over the chosen set:  dl_j = g_j (dg_j - sum_i g_i dg_i)
    sigmoid, normalised:          ds_j = (dg_j - sum_i g_i dg_i) / sum_S sig,
                                  dl_j = ds_j sig_j (1 - sig_j)
    """
    logits = np.asarray(logits, np.float64)
    sel = np.asarray(sel, np.int64)
    g = np.asarray(gates, np.float64)
    dg = np.asarray(dgate, np.float64)
    inner = (g * dg).sum(axis=-1, keepdims=True)
    if score == SOFTMAX:
        dl_sel = g * (dg - inner)
    elif score == SIGMOID:
        l_sel = np.take_along_axis(logits, sel, axis=-1)
        s = _sigmoid(l_sel)
        ds = (dg - inner) / s.sum(axis=-1, keepdims=True)
        dl_sel = ds * s * (1.0 - s)
    else:
        raise ValueError(score)
    dlogits = np.zeros_like(logits)
    np.put_along_axis(dlogits, sel, dl_sel, axis=-1)
    return dlogits


def moe_backward(x, w_router, w1, w2, fwd, dy, score=SOFTMAX,
                 w1_shared=None, w2_shared=None, with_router=True, weight_grads=True):
    """Gradients of L = <dy, y> with the routing held fixed (top-k is piecewise
    constant), by the chain rule, in fp64.

    Per routed pair (t,i), e = S_t[i], z = W1_e x_t = [a, b], h = silu(a) * b:
      dgate[t,i] = <dy_t, W2_e h>
      dh  = g * W2_e^T dy_t;  da = dh * b * silu'(a);  db = dh * silu(a)
      dx_t += W1_e^T [da, db];  dW1_e += [da, db] x_t^T;  dW2_e += dy_t (g h)^T
    Router: dlogits = router_backward(...); dx_t += Wr^T dl_t; dWr += dl_t x_t^T.
    Shared expert: the same with g = 1 and no gate gradient.
    weight_grads=False leaves out dW1, dW2, dWr and the shared expert's
    weight gradients (for large layers evaluated on a few tokens).
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    T, H = x.shape
    E = _shape(w1)[0]
    F = _shape(w1)[1] // 2
    idx = np.asarray(fwd["topk_idx"], np.int64)
    gate = np.asarray(fwd["gates"], np.float64)
    k = idx.shape[1]
    dx = np.zeros_like(x)
    dW1 = np.zeros((E, 2 * F, H)) if weight_grads else None
    dW2 = np.zeros((E, H, F)) if weight_grads else None
    dgate = np.zeros((T, k))
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        W1 = np.asarray(w1[e], np.float64)
        W2 = np.asarray(w2[e], np.float64)
        xe = x[tok]
        z = xe @ W1.T
        a, b = z[:, :F], z[:, F:]
        h = silu(a) * b
        g = gate[tok, slot][:, None]
        dye = dy[tok]
        dgate[tok, slot] = ((dye @ W2) * h).sum(axis=1)
        dh = g * (dye @ W2)
        da = dh * b * silu_grad(a)
        db = dh * silu(a)
        dz = np.concatenate([da, db], axis=1)
        np.add.at(dx, tok, dz @ W1)
        if weight_grads:
            dW1[e] = dz.T @ xe
            dW2[e] = dye.T @ (g * h)
    out = {"dx": dx, "dgate": dgate}
    if weight_grads:
        out.update(dW1=dW1, dW2=dW2)
    if w1_shared is not None:
        W1 = np.asarray(w1_shared, np.float64)
        W2 = np.asarray(w2_shared, np.float64)
        S = W1.shape[0] // 2
        z = x @ W1.T
        a, b = z[:, :S], z[:, S:]
        h = silu(a) * b
        dh = dy @ W2
        dz = np.concatenate([dh * b * silu_grad(a), dh * silu(a)], axis=1)
        dx += dz @ W1
        if weight_grads:
            out["dW1_shared"] = dz.T @ x
            out["dW2_shared"] = dy.T @ h
    if with_router:
        logits = fwd["logits"] if fwd.get("logits") is not None else router_logits(x, w_router)
        dl = router_backward(logits, idx, gate, dgate, score)
        dx += dl @ np.asarray(w_router, np.float64)
        out["dlogits"] = dl
        if weight_grads:
            out["dWr"] = dl.T @ x
    out["dx"] = dx
    return out


# ---------------------------------------------------------------------------
# MXFP8: OCP Microscaling v1.0 (E8M0 block scale, 32 elements) with the
# FP8 E4M3 element type (OCP 8-bit floating point v1.0: bias 7, no infinities,
# largest finite 448, S.1111.111 is NaN).  Technical summary 2.5 names MXFP8 as
# the Blackwell recipe; the block size 32 and element type are the MX format's.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0
MX_BLOCK = 32
E4M3_EMAX = 8          # exponent of the largest normal power of two, 2^8 = 256


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 bit pattern (uint8) as fp64; 0x7F / 0xFF give NaN."""
    c = np.asarray(code, np.int64) & 0xFF
    s = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ex == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(ex.astype(np.float64) - 7.0))
    val = np.where((ex == 15) & (m == 7), np.nan, val)
    return s * val


def _round_half_even(v: np.ndarray) -> np.ndarray:
    return np.round(v)          # numpy rounds halves to even


def e4m3_encode(v) -> np.ndarray:
    """Round fp64 values to E4M3, nearest-even, saturating to +-448 (the
    'satfinite' behaviour).  Returns uint8 bit patterns.  Inputs must be finite."""
    v = np.asarray(v, np.float64)
    sign = np.signbit(v)
    a = np.abs(v)
    # quantisation step: 2^(p-3) for |v| in [2^p, 2^(p+1)), p >= -6; 2^-9 below 2^-6
    _, p1 = np.frexp(a)                    # a = f * 2^p1, f in [0.5, 1)
    p = np.maximum(p1 - 1, -6)
    step = np.exp2((p - 3).astype(np.float64))
    q = _round_half_even(a / step) * step
    q = np.minimum(q, E4M3_MAX)
    # encode q (now exactly representable)
    _, qp1 = np.frexp(q)
    qp = qp1 - 1
    normal = q >= 2.0 ** -6
    ex = np.where(normal, qp + 7, 0)
    mant = np.where(normal, q / np.exp2(qp.astype(np.float64)) * 8.0 - 8.0, q / 2.0 ** -9)
    code = (ex.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(q == 0, 0, code)
    code = code | np.where(sign, 0x80, 0)
    return code.astype(np.uint8)


def mx_scale_exponent(amax) -> np.ndarray:
    """Shared exponent of a block: floor(log2(amax)) - 8, clamped to E8M0's
    range [-127, 127]; amax == 0 gives -127.  The X = 2^e rule of OCP MX v1.0
    (the largest element lands in E4M3's top binade)."""
    amax = np.asarray(amax, np.float64)
    _, p1 = np.frexp(amax)
    e = (p1 - 1) - E4M3_EMAX
    e = np.where(amax == 0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def mxfp8_quantize(v, axis=-1):
    """Quantise along ``axis`` in blocks of 32: returns (codes uint8, same shape;
    scales uint8 E8M0 = exponent + 127, with the blocked axis divided by 32).
    q = e4m3(v / 2^e) with e = mx_scale_exponent(max |v| over the block)."""
    v = np.moveaxis(np.asarray(v, np.float64), axis, -1)
    shp = v.shape
    if shp[-1] % MX_BLOCK:
        raise ValueError("blocked axis must be a multiple of 32")
    blocks = v.reshape(shp[:-1] + (shp[-1] // MX_BLOCK, MX_BLOCK))
    e = mx_scale_exponent(np.abs(blocks).max(axis=-1))
    scaled = blocks / np.exp2(e.astype(np.float64))[..., None]
    codes = e4m3_encode(scaled).reshape(shp)
    scales = (e + 127).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mxfp8_dequantize(codes, scales, axis=-1):
    """Inverse map: value = e4m3(code) * 2^(scale - 127), block of 32 along axis."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1).astype(np.float64)
    vals = e4m3_decode(c)
    rep = np.repeat(np.exp2(s - 127.0), MX_BLOCK, axis=-1)
    return np.moveaxis(vals * rep, -1, axis)


def mxfp8_roundtrip(v, axis=-1):
    """dequantize(quantize(v)) along axis: the operand an MXFP8 GEMM multiplies."""
    c, s = mxfp8_quantize(v, axis)
    return mxfp8_dequantize(c, s, axis)


# ---------------------------------------------------------------------------
# Step-level definitions in the expert-ordered (padded) row layout.  Each one
# is the plain definition of one grouped step, expert by expert; composing
# them gives moe_forward / moe_backward (pinned in tests/test_oracle_steps.py).
# Rows of expert e: [poffsets[e], poffsets[e+1]), padding rows included.
# ---------------------------------------------------------------------------

def _segments(poffsets):
    po = np.asarray(poffsets, np.int64)
    return [(e, int(po[e]), int(po[e + 1])) for e in range(len(po) - 1)]


def expert_fc1(x_perm, w1, poffsets, row_gate=None):
    """z_r = W1_e x_r for each row r of expert e; h_r = g_r * silu(z_gate) * z_up
    (the routing weight applied at the activation, technical summary 2.2)."""
    x_perm = np.asarray(x_perm, np.float64)
    F = _shape(w1)[1] // 2
    rows = x_perm.shape[0]
    z = np.zeros((rows, 2 * F))
    for e, a, b in _segments(poffsets):
        if b > a:
            z[a:b] = x_perm[a:b] @ np.asarray(w1[e], np.float64).T
    g = np.ones(rows) if row_gate is None else np.asarray(row_gate, np.float64)
    h = g[:, None] * silu(z[:, :F]) * z[:, F:]
    return z, h


def expert_fc2(h, w2, poffsets):
    """o_r = W2_e h_r."""
    h = np.asarray(h, np.float64)
    H = _shape(w2)[1]
    o = np.zeros((h.shape[0], H))
    for e, a, b in _segments(poffsets):
        if b > a:
            o[a:b] = h[a:b] @ np.asarray(w2[e], np.float64).T
    return o


def expert_dgrad_fc2(dy_perm, w2, z, poffsets, row_gate=None):
    """dh'_r = W2_e^T dy_r; with a, b = z_r halves:  dgate_r = <dh'_r, silu(a) b>,
    dz_r = [g dh' b silu'(a), g dh' silu(a)].  Returns (dz, dgate_rows)."""
    dy_perm = np.asarray(dy_perm, np.float64)
    z = np.asarray(z, np.float64)
    F = z.shape[1] // 2
    rows = dy_perm.shape[0]
    dhp = np.zeros((rows, F))
    for e, a, b in _segments(poffsets):
        if b > a:
            dhp[a:b] = dy_perm[a:b] @ np.asarray(w2[e], np.float64)
    za, zb = z[:, :F], z[:, F:]
    g = np.ones(rows) if row_gate is None else np.asarray(row_gate, np.float64)
    dgate_rows = (dhp * silu(za) * zb).sum(axis=1)
    dh = g[:, None] * dhp
    dz = np.concatenate([dh * zb * silu_grad(za), dh * silu(za)], axis=1)
    return dz, dgate_rows


def expert_dgrad_fc1(dz, w1, poffsets):
    """dx_r = W1_e^T dz_r."""
    dz = np.asarray(dz, np.float64)
    H = _shape(w1)[2]
    dx = np.zeros((dz.shape[0], H))
    for e, a, b in _segments(poffsets):
        if b > a:
            dx[a:b] = dz[a:b] @ np.asarray(w1[e], np.float64)
    return dx


def expert_wgrad(a_rows, b_rows, poffsets):
    """dW_e = sum over expert e's rows of a_r b_r^T ([E, M, N]; zero for empty experts)."""
    A = np.asarray(a_rows, np.float64)
    B = np.asarray(b_rows, np.float64)
    segs = _segments(poffsets)
    out = np.zeros((len(segs), A.shape[1], B.shape[1]))
    for e, a, b in segs:
        if b > a:
            out[e] = A[a:b].T @ B[a:b]
    return out


def dense_rows_of(n_rows):
    """poffsets of one group holding rows [0, n_rows) (the shared expert)."""
    return np.array([0, n_rows], np.int64)


# ---------------------------------------------------------------------------
# The layer under the MXFP8 recipe (technical summary 2.5: expert GEMMs and
# their activations in FP8 with MX block scales; router, gates, combine in
# high precision).  Each expert-GEMM operand passes through the MX quantiser
# along that GEMM's contraction axis (blocks of 32 consecutive values):
#   fc1:       x rows along H,  W1_e along H
#   fc2:       h' = g*silu(a)*b along F (the gate is applied before the
#              quantiser, as the layer applies it inside fc1), W2_e along F
#   fc2 dgrad: dy rows along H, W2_e along H
#   fc1 dgrad: dz rows along 2F, W1_e along 2F
#   wgrad:     dz, x, dy, h' along the tokens of the expert, in expert order
#              (ascending token), zero-padded to whole blocks
# ``quant(v, axis)`` is the quantise-dequantise map; the identity gives back
# the unquantised layer (tests/test_oracle_mx.py pins that).
# ---------------------------------------------------------------------------

def _pad_rows(a, mult=32):
    r = a.shape[0]
    p = (-r) % mult
    if p == 0:
        return a
    return np.concatenate([a, np.zeros((p,) + a.shape[1:])], axis=0)


def _q_tokens(a, quant):
    """Quantise along the token axis in blocks of 32 rows (zero padding)."""
    r = a.shape[0]
    return quant(_pad_rows(a), 0)[:r]


def _weight_quantiser(quant, cache):
    """quant for weights, memoised in ``cache`` (a dict) by (tensor, expert, axis):
    the recipe quantises each weight once, so repeated calls may reuse it."""
    if cache is None:
        return lambda name, e, W, axis: quant(W, axis)

    def qw(name, e, W, axis):
        key = (name, e, axis)
        if key not in cache:
            cache[key] = quant(W, axis)
        return cache[key]
    return qw


def moe_forward_mx(x, w_router, w1, w2, k, score=SOFTMAX, bias=None, w1_shared=None, w2_shared=None,
                   routing=None, quant=mxfp8_roundtrip, weight_cache=None):
    qw = _weight_quantiser(quant, weight_cache)
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = _shape(w1)[0]
    F = _shape(w1)[1] // 2
    logits = None
    if routing is None:
        logits = router_logits(x, w_router)
        idx, gate = route(logits, k, score, bias)
    else:
        idx = np.asarray(routing[0], np.int64)
        gate = np.asarray(routing[1], np.float64)
    y = np.zeros_like(x)
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        W1 = np.asarray(w1[e], np.float64)
        W2 = np.asarray(w2[e], np.float64)
        z = quant(x[tok], -1) @ qw("w1", e, W1, -1).T
        hp = gate[tok, slot][:, None] * silu(z[:, :F]) * z[:, F:]
        np.add.at(y, tok, quant(hp, -1) @ qw("w2", e, W2, -1).T)
    if w1_shared is not None:
        W1 = np.asarray(w1_shared, np.float64)
        W2 = np.asarray(w2_shared, np.float64)
        S = W1.shape[0] // 2
        z = quant(x, -1) @ qw("w1s", 0, W1, -1).T
        y += quant(silu(z[:, :S]) * z[:, S:], -1) @ qw("w2s", 0, W2, -1).T
    return {"y": y, "logits": logits, "topk_idx": idx.astype(np.int32), "gates": gate}


def moe_backward_mx(x, w_router, w1, w2, fwd, dy, score=SOFTMAX, w1_shared=None, w2_shared=None,
                    quant=mxfp8_roundtrip, weight_cache=None, weight_grads=True):
    """Gradients as the MXFP8 recipe computes them: the chain rule of the
    unquantised layer, with every expert-GEMM operand quantised along its
    contraction axis (straight through the quantiser).  weight_grads=False
    leaves out the weight gradients, as in moe_backward."""
    qw = _weight_quantiser(quant, weight_cache)
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    T, H = x.shape
    E = _shape(w1)[0]
    F = _shape(w1)[1] // 2
    idx = np.asarray(fwd["topk_idx"], np.int64)
    gate = np.asarray(fwd["gates"], np.float64)
    k = idx.shape[1]
    dx = np.zeros_like(x)
    dW1 = np.zeros((E, 2 * F, H)) if weight_grads else None
    dW2 = np.zeros((E, H, F)) if weight_grads else None
    dgate = np.zeros((T, k))
    for e in range(E):
        tok, slot = np.nonzero(idx == e)          # ascending token: the expert's row order
        if tok.size == 0:
            continue
        W1 = np.asarray(w1[e], np.float64)
        W2 = np.asarray(w2[e], np.float64)
        xe = x[tok]
        z = quant(xe, -1) @ qw("w1", e, W1, -1).T
        a, b = z[:, :F], z[:, F:]
        h = silu(a) * b
        g = gate[tok, slot][:, None]
        dye = dy[tok]
        dhp = quant(dye, -1) @ qw("w2", e, W2, 0)           # contraction over H
        dgate[tok, slot] = (dhp * h).sum(axis=1)
        dh = g * dhp
        dz = np.concatenate([dh * b * silu_grad(a), dh * silu(a)], axis=1)
        np.add.at(dx, tok, quant(dz, -1) @ qw("w1", e, W1, 0))  # contraction over 2F
        if weight_grads:
            dW1[e] = _q_tokens(dz, quant).T @ _q_tokens(xe, quant)
            dW2[e] = _q_tokens(dye, quant).T @ _q_tokens(g * h, quant)
    out = {"dgate": dgate}
    if weight_grads:
        out.update(dW1=dW1, dW2=dW2)
    if w1_shared is not None:
        W1 = np.asarray(w1_shared, np.float64)
        W2 = np.asarray(w2_shared, np.float64)
        S = W1.shape[0] // 2
        z = quant(x, -1) @ qw("w1s", 0, W1, -1).T
        a, b = z[:, :S], z[:, S:]
        h = silu(a) * b
        dh = quant(dy, -1) @ qw("w2s", 0, W2, 0)
        dz = np.concatenate([dh * b * silu_grad(a), dh * silu(a)], axis=1)
        dx += quant(dz, -1) @ qw("w1s", 0, W1, 0)
        if weight_grads:
            out["dW1_shared"] = _q_tokens(dz, quant).T @ _q_tokens(x, quant)
            out["dW2_shared"] = _q_tokens(dy, quant).T @ _q_tokens(h, quant)
    logits = fwd["logits"] if fwd.get("logits") is not None else router_logits(x, w_router)
    dl = router_backward(logits, idx, gate, dgate, score)
    dx += dl @ np.asarray(w_router, np.float64)
    out["dlogits"] = dl
    if weight_grads:
        out["dWr"] = dl.T @ x
    out["dx"] = dx
    return out


# ---------------------------------------------------------------------------
# NVFP4 expert GEMMs (technical summary 2.5: NVFP4 named beside MXFP8 as a
# Blackwell quantisation recipe for the expert GEMMs and activations).  The
# pages give no recipe; the reading taken is the NVFP4 format itself:
#   * elements FP4 E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit:
#     0, 0.5, 1, 1.5, 2, 3, 4, 6), rounded to nearest even, saturated to +-6;
#   * one unsigned E4M3 scale per block of 16 consecutive values along the
#     contraction;
#   * one fp32 scale per tensor from its largest magnitude, so the block scales
#     land in E4M3's range: S = 2688 / amax (2688 = 6 * 448, the E2M1 and E4M3
#     maxima).
# The encoding decisions (scale byte, element codes) are taken in fp32 in the
# order written below, the precision the GPU quantiser works in, so both sides
# make the same decisions from the same bf16 inputs:
#   s_f  = fp32(fp32(amax_b / 6) * S)       block scale before rounding
#   s    = e4m3(s_f)                        (round to nearest even, satfinite)
#   r    = fp32(S / s)  (0 when s == 0)     multiplier of the block's values
#   code = e2m1(fp32(v * r))
# and a value is decoded as e2m1(code) * s / S.  S and r are capped at the
# largest finite fp32 (only reached for tensors with amax below ~1e-33).
# ---------------------------------------------------------------------------

E2M1_MAX = 6.0
NV_BLOCK = 16
NV_TENSOR_RANGE = 2688.0     # E2M1 max * E4M3 max
_F32_MAX = float(np.finfo(np.float32).max)


def e2m1_decode(code) -> np.ndarray:
    """Value of each 4-bit E2M1 pattern (low nibble of the input) as fp64."""
    c = np.asarray(code, np.int64) & 0xF
    s = np.where(c & 0x8, -1.0, 1.0)
    ex = (c >> 1) & 0x3
    m = c & 0x1
    val = np.where(ex == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(ex.astype(np.float64) - 1.0))
    return s * val


def e2m1_encode(v) -> np.ndarray:
    """Round fp64 values to E2M1, nearest-even, saturating to +-6.  Returns the
    4-bit patterns as uint8.  Inputs must be finite."""
    v = np.asarray(v, np.float64)
    sign = np.signbit(v)
    a = np.minimum(np.abs(v), E2M1_MAX)
    # quantisation step: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = np.minimum(_round_half_even(a / step) * step, E2M1_MAX)
    # encode q (exactly representable): subnormal 0.5 -> 0b001, else exponent/mantissa
    _, qp1 = np.frexp(q)
    qp = qp1 - 1
    normal = q >= 1.0
    ex = np.where(normal, qp + 1, 0)
    mant = np.where(normal, q / np.exp2(qp.astype(np.float64)) * 2.0 - 2.0, q / 0.5)
    code = (ex.astype(np.int64) << 1) | mant.astype(np.int64)
    code = np.where(q == 0, 0, code) | np.where(sign, 0x8, 0)
    return code.astype(np.uint8)


def nvfp4_tensor_scale(amax) -> np.float32:
    """S = 2688 / amax in fp32 (1 for an all-zero tensor), capped at the largest fp32."""
    amax = np.float32(amax)
    if not amax > 0:
        return np.float32(1.0)
    with np.errstate(over="ignore"):
        s = np.float32(NV_TENSOR_RANGE) / amax
    return np.float32(min(float(s), _F32_MAX))


def nvfp4_quantize(v, amax=None, axis=-1):
    """Quantise along ``axis`` in blocks of 16 with the tensor scale of ``amax``
    (default: max |v| over the whole array).  Returns (codes uint8 holding one
    E2M1 pattern each, same shape as v; scales uint8 E4M3 with the blocked
    axis divided by 16).  v is taken in fp32 (bf16 inputs are exact there)."""
    v32 = np.moveaxis(np.asarray(v, np.float32), axis, -1)
    if amax is None:
        amax = np.abs(v32).max() if v32.size else 0.0
    S = nvfp4_tensor_scale(amax)
    shp = v32.shape
    if shp[-1] % NV_BLOCK:
        raise ValueError("blocked axis must be a multiple of 16")
    blocks = v32.reshape(shp[:-1] + (shp[-1] // NV_BLOCK, NV_BLOCK))
    amax_b = np.abs(blocks).max(axis=-1)
    s_f = (amax_b / np.float32(6.0)).astype(np.float32) * S           # fp32 divide, fp32 multiply
    s_code = e4m3_encode(s_f.astype(np.float64))
    s_val = e4m3_decode(s_code).astype(np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        r = np.where(s_val > 0, S / np.where(s_val > 0, s_val, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    r = np.minimum(r, np.float32(_F32_MAX))
    scaled = (blocks * r[..., None]).astype(np.float32)
    codes = e2m1_encode(scaled.astype(np.float64)).reshape(shp)
    return np.moveaxis(codes, -1, axis), np.moveaxis(s_code, -1, axis), S


def nvfp4_dequantize(codes, scales, S, axis=-1):
    """value = e2m1(code) * e4m3(scale) / S, one scale per 16 along axis."""
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    rep = np.repeat(e4m3_decode(s), NV_BLOCK, axis=-1)
    return np.moveaxis(e2m1_decode(c) * rep / np.float64(S), -1, axis)


def nvfp4_roundtrip(v, amax=None, axis=-1):
    """dequantize(quantize(v)): the operand an NVFP4 GEMM multiplies."""
    c, s, S = nvfp4_quantize(v, amax, axis)
    return nvfp4_dequantize(c, s, S, axis)


def bf16_round(v) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as fp64: the
    storage type of the activations the quantiser reads."""
    f = np.ascontiguousarray(np.asarray(v, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def nvfp4_weight(cache, name, W, e=None, quant=nvfp4_roundtrip):
    """Quantise-dequantise expert e of the weight tensor W (or all of a 2-D W
    when e is None) with the tensor amax over every expert, memoised in
    ``cache`` (a dict): the recipe quantises each weight once.  W may be any
    object whose W[e] gives expert e as an array."""
    key = (name, e)
    if key not in cache:
        akey = (name, "amax")
        if akey not in cache:
            if e is None:
                cache[akey] = float(np.abs(np.asarray(W, np.float32)).max())
            else:
                cache[akey] = max(float(np.abs(np.asarray(W[i], np.float32)).max()) for i in range(_shape(W)[0]))
        Wi = W if e is None else W[e]
        cache[key] = quant(np.asarray(Wi, np.float64), cache[akey], -1)
    return cache[key]


def moe_forward_nvfp4(x, w_router, w1, w2, k, score=SOFTMAX, bias=None, w1_shared=None, w2_shared=None,
                      routing=None, weight_cache=None, quant=nvfp4_roundtrip, store=bf16_round,
                      x_amax=None, h_amax=None):
    """Forward with NVFP4 expert GEMMs.  Each quantised tensor has its own
    tensor scale: x (all tokens), W1 and W2 (all experts), h' (the gated
    activation of every expert row, rounded to bf16 as it is stored), and the
    shared expert's W1s, W2s and h.  Everything else as moe_forward.
    ``quant(v, amax, axis)`` and ``store(v)`` are the quantise-dequantise map
    and the activation storage rounding; identities give back the unquantised
    layer (tests/test_oracle_nvfp4.py pins that).  ``x_amax`` / ``h_amax``
    replace the tensor amaxes of x and h' when x holds only some of the
    tokens (every other step is row-local, so those rows then come out as in
    the forward of all tokens)."""
    x = np.asarray(x, np.float64)
    E = _shape(w1)[0]
    F = _shape(w1)[1] // 2
    cache = weight_cache if weight_cache is not None else {}

    def wq(name, W, e):
        return nvfp4_weight(cache, name, W, e, quant)

    logits = None
    if routing is None:
        logits = router_logits(x, w_router)
        idx, gate = route(logits, k, score, bias)
    else:
        idx = np.asarray(routing[0], np.int64)
        gate = np.asarray(routing[1], np.float64)
    xq = quant(x, x_amax, -1)
    rows = []
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        z = xq[tok] @ wq("w1", w1, e).T
        hp = store(gate[tok, slot][:, None] * silu(z[:, :F]) * z[:, F:])
        rows.append((e, tok, hp))
    amax_h = max((np.abs(hp).max() for _, _, hp in rows), default=0.0) if h_amax is None else h_amax
    y = np.zeros_like(x)
    for e, tok, hp in rows:
        np.add.at(y, tok, quant(hp, amax_h, -1) @ wq("w2", w2, e).T)
    if w1_shared is not None:
        W1s, W2s = wq("w1s", w1_shared, None), wq("w2s", w2_shared, None)
        S = W1s.shape[0] // 2
        z = xq @ W1s.T
        hs = store(silu(z[:, :S]) * z[:, S:])
        y += quant(hs, None, -1) @ W2s.T
    return {"y": y, "logits": logits, "topk_idx": idx.astype(np.int32), "gates": gate}
