"""Plain CPU oracle of the single-GPU Mixture-of-Experts layer.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg use this module. It shares no code with the CUDA library and
imports nothing from it; the CUDA library never calls it.

Every step is written out as its plain definition in float64 (storage of the
inputs is whatever the caller passes: fp32 values, or bf16 values read as
floats). Library primitives used as single steps: numpy matmul, stable argsort,
bincount, cumsum. No blocking, fusion or reordering beyond what each definition
states.

Sources. Three web pages describe the method:
  [warp] "Cursor a réécrit le décodage de MoE" (toolnavs.com), sections
         "Cursor a réécrit le décodage de MoE" and "1.84x plus de vitesse ...":
         small-batch decode where each warp owns one output value, two kernels.
  [MoK]  "Cursor открыл код ядра Mixture of Experts: обучение MoE ускоряется
         до 2,37 раза" (dzen.guru), sections "Что именно тормозило обучение
         MoE-моделей?" (each layer routes tokens to experts, runs them, gathers
         the results back) and "Три решения, которые дали результат" (pull
         dispatch, push combine, fixed ring buffer walked in reverse in the
         backward pass, deterministic result, BF16 and MXFP8).
  [kittens] the khabar-ai page quoting the Mixture-of-Kittens release thread.
The pages print no formula. The layer math below (top-k router with softmax or
sigmoid gates renormalised over the selected experts, SwiGLU experts, shared
expert, weighted combine) is the standard MoE layer those pages refer to; each
point where they are silent is resolved by the plainest reading, noted inline.

Pins: every function here is checked by the CPU tests against brute force on
tiny inputs, closed forms, invariants and hand-derived golden values.
"""
from __future__ import annotations

import numpy as np

f64 = np.float64


# --------------------------------------------------------------------------
# Router  [MoK, "Что именно тормозило ...": each layer routes tokens to experts]
# --------------------------------------------------------------------------

def router_logits(x, Wr):
    """l[t, e] = sum_i x[t, i] * Wr[e, i]  (float64)."""
    return np.asarray(x, f64) @ np.asarray(Wr, f64).T


def selection_keys(logits32, bias32):
    """Selection key = l + b, formed in fp32 like the GPU kernel forms it.

    The bias enters the selection only (reading: a load-balancing bias in logit
    space, added to the fp32 logits); gates use the unbiased logits.
    """
    l32 = np.asarray(logits32, np.float32)
    b32 = np.asarray(bias32, np.float32)
    return (l32 + b32[None, :]).astype(np.float32)


def select_experts(logits32, bias32, k: int):
    """idx[t, j]: the k largest keys of token t, largest first; ties go to the lower expert.

    Reading: slot order j is (key descending, expert ascending). A stable sort of
    the negated keys gives exactly that order.
    """
    key = selection_keys(logits32, bias32)
    order = np.argsort(-key, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gates_softmax(logits, idx, renorm: bool = True):
    """Softmax gates. renorm: softmax over the k selected logits; else softmax over all E, taken at idx."""
    l = np.asarray(logits, f64)
    if renorm:
        sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
        m = sel.max(axis=1, keepdims=True)
        ex = np.exp(sel - m)
        return ex / ex.sum(axis=1, keepdims=True)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    p = p / p.sum(axis=1, keepdims=True)
    return np.take_along_axis(p, idx.astype(np.int64), axis=1)


def sigmoid(z):
    z = np.asarray(z, f64)
    return 1.0 / (1.0 + np.exp(-z))


def gates_sigmoid(logits, idx, scale: float, renorm: bool = True):
    """Sigmoid gates s = 1/(1+exp(-l)) at the selected experts; renorm: scale * s / sum(s)."""
    sel = np.take_along_axis(np.asarray(logits, f64), idx.astype(np.int64), axis=1)
    s = sigmoid(sel)
    if renorm:
        return scale * s / s.sum(axis=1, keepdims=True)
    return scale * s


def gates(logits, idx, router: str, renorm: bool, scale: float):
    if router == "softmax":
        return scale * gates_softmax(logits, idx, renorm) if scale != 1.0 else gates_softmax(logits, idx, renorm)
    if router == "sigmoid":
        return gates_sigmoid(logits, idx, scale, renorm)
    raise ValueError(router)


# --------------------------------------------------------------------------
# Dispatch bookkeeping  [MoK, "Три решения ...": dropless, no CPU-sized buffers]
# --------------------------------------------------------------------------

def expert_counts(idx, E: int):
    """cnt[e] = number of (token, slot) assignments routed to expert e. Dropless: sum = T*k."""
    return np.bincount(np.asarray(idx).ravel().astype(np.int64), minlength=E).astype(np.int64)


def expert_offsets(cnt):
    """Exclusive prefix sum: off[e] = sum_{e' < e} cnt[e'], off[E] = total."""
    return np.concatenate([[0], np.cumsum(cnt)]).astype(np.int64)


def stable_permutation(idx):
    """perm[p] = assignment a = t*k + j at sorted position p, sorted by (expert, a); inv = perm^-1.

    Reading: within an expert, assignments keep ascending a (the unique order
    that does not depend on any schedule).
    """
    flat = np.asarray(idx).ravel().astype(np.int64)
    perm = np.argsort(flat, kind="stable")
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return perm, inv


def permute_rows(X, perm, k: int):
    """Rows of X (one per token) in sorted assignment order: row p is X[perm[p] // k]."""
    return np.asarray(X)[np.asarray(perm) // k]


def unpermute_rows(Y, inv):
    """Rows in assignment order: row a is Y[inv[a]]."""
    return np.asarray(Y)[np.asarray(inv)]


# --------------------------------------------------------------------------
# Expert FFN (SwiGLU)
# --------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, f64)
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d/dz silu(z) = sigma(z) * (1 + z * (1 - sigma(z)))."""
    s = sigmoid(z)
    return s * (1.0 + np.asarray(z, f64) * (1.0 - s))


def expert_ffn(xr, Wg_e, Wu_e, Wd_e):
    """o = (silu(x Wg^T) * (x Wu^T)) Wd^T for the rows xr. Returns (u, v, h, o)."""
    xr = np.asarray(xr, f64)
    u = xr @ np.asarray(Wg_e, f64).T
    v = xr @ np.asarray(Wu_e, f64).T
    h = silu(u) * v
    o = h @ np.asarray(Wd_e, f64).T
    return u, v, h, o


# --------------------------------------------------------------------------
# MXFP8 quantiser (OCP Microscaling Formats v1.0: E4M3 elements, E8M0 scale per 32)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal E4M3 value (448 = 1.75 * 2^8)
E4M3_EMIN = -6         # smallest normal exponent; subnormals are m * 2^-9, m = 1..7
E4M3_MBITS = 3


def e4m3_round(v):
    """Round reals to the nearest E4M3 value (ties to even), saturating at +-448 (sign kept, -0 stays -0)."""
    v = np.asarray(v, f64)
    a = np.abs(v)
    ex = np.frexp(a)[1] - 1                  # a in [2^ex, 2^(ex+1))
    e = np.maximum(ex, E4M3_EMIN)            # subnormals share the 2^-6 binade's quantum
    quantum = np.ldexp(1.0, e - E4M3_MBITS)
    q = np.round(a / quantum) * quantum      # np.round rounds halves to even; a/quantum is exact
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode(q):
    """Bit patterns (sign, 4-bit exponent with bias 7, 3-bit mantissa) of E4M3 values."""
    q = np.asarray(q, f64)
    sign = np.where(np.signbit(q), 0x80, 0)
    a = np.abs(q)
    e = np.frexp(a)[1] - 1
    sub = a < 2.0 ** E4M3_EMIN
    m_sub = np.rint(a / 2.0 ** -9).astype(np.int64)
    e_n = np.where(sub, 0, e)
    m_n = np.rint(a / np.ldexp(1.0, e_n - 3)).astype(np.int64) - 8
    code = np.where(sub, m_sub, ((e_n + 7) << 3) | (m_n & 7))
    return (sign | code).astype(np.uint8)


def e4m3_decode_scalar(byte: int) -> float:
    """Value of one E4M3 bit pattern (S.EEEE.MMM, bias 7; S.1111.111 is NaN)."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 7
    if e == 0:
        return s * m * 2.0 ** -9
    if e == 15 and m == 7:
        return float("nan")
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_TABLE = np.array([e4m3_decode_scalar(b) for b in range(256)], f64)


def e4m3_decode(codes):
    return _E4M3_TABLE[np.asarray(codes, np.uint8)]


def mx_block_scale_exponent(amax):
    """Shared exponents X = floor(log2(amax)) - 8, clamped to [-127, 127]; amax = 0 gives -127."""
    amax = np.asarray(amax, f64)
    X = np.frexp(amax)[1] - 1 - E4M3_EMAX
    X = np.clip(X, -127, 127)
    return np.where(amax == 0.0, -127, X).astype(np.int64)


def mx_quantize(a, axis: int = -1, block: int = 32):
    """Quantise along `axis` in blocks of 32: returns (E4M3 codes uint8, E8M0 scales uint8).

    codes has the shape of a; scales has a's shape with `axis` divided by 32.
    Element value = decode(code) * 2^(scale - 127).
    """
    a = np.moveaxis(np.asarray(a, f64), axis, -1)
    n = a.shape[-1]
    if n % block:
        raise ValueError("length along the quantised axis must be a multiple of 32")
    blk = a.reshape(a.shape[:-1] + (n // block, block))
    X = mx_block_scale_exponent(np.max(np.abs(blk), axis=-1))
    scaled = blk * np.ldexp(1.0, -X)[..., None]     # exact: a power-of-two scaling
    codes = e4m3_encode(e4m3_round(scaled)).reshape(a.shape)
    scales = (X + 127).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mx_dequantize(codes, scales, axis: int = -1, block: int = 32):
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1).astype(np.int64)
    vals = e4m3_decode(c)
    mult = np.ldexp(1.0, s - 127)
    out = vals * np.repeat(mult, block, axis=-1)
    return np.moveaxis(out, -1, axis)


def mx_fake_quant(a, axis: int = -1):
    """The values an MXFP8 tensor holds after quantising a along axis (exact dequantisation)."""
    codes, scales = mx_quantize(a, axis)
    return mx_dequantize(codes, scales, axis)


# --------------------------------------------------------------------------
# Forward  [MoK: route, dispatch (pull), experts, combine (push); deterministic]
# --------------------------------------------------------------------------

def route(x, Wr, b, k: int, router: str, renorm: bool, scale: float, logits32=None):
    """Router logits, top-k selection, gates, counts, offsets and the stable permutation.

    logits32 (optional): route these fp32 logits instead of computing them (the
    bit-exact routing comparison feeds the GPU's logits here).
    """
    if logits32 is None:
        l = router_logits(x, Wr)
    else:
        l = np.asarray(logits32, np.float32).astype(f64)
    E = np.asarray(Wr).shape[0]
    # the selection is an integer decision taken in fp32, as the kernel takes it;
    # the gates use the float64 logits
    idx = select_experts(l.astype(np.float32), b, k)
    g = gates(l, idx, router, renorm, scale)
    cnt = expert_counts(idx, E)
    off = expert_offsets(cnt)
    perm, inv = stable_permutation(idx)
    return dict(logits=l, idx=idx, gate=g, cnt=cnt, off=off, perm=perm, inv=inv)


def forward(x, Wr, b, Wg, Wu, Wd, k: int, router: str, renorm: bool, scale: float,
            n_shared: int = 0, logits32=None, mx: bool = False, keep: bool = False):
    """y[t] = shared(x_t) + sum_j gate[t, j] * FFN_{idx[t, j]}(x_t), summed shared first then j = 0..k-1.

    Reading: the shared expert has gate 1 and is not scaled. mx=True: x and the
    weights are fake-quantised along each GEMM's K and h is quantised along f
    before the down projection, as an MXFP8 layer does.
    """
    x = np.asarray(x, f64)
    T, d = x.shape
    E = np.asarray(Wr).shape[0]
    r = route(x, Wr, b, k, router, renorm, scale, logits32)
    idx, g, perm, off = r["idx"], r["gate"], r["perm"], r["off"]
    if mx:
        xq = mx_fake_quant(x, axis=1)
    else:
        xq = x
    o = np.zeros((T * k, d), f64)            # expert output per assignment a = t*k + j
    u_all = v_all = None
    if keep:
        f = np.asarray(Wg).shape[1]
        u_all = np.zeros((T * k, f), f64)
        v_all = np.zeros((T * k, f), f64)
    for e in range(E):
        rows = perm[off[e]:off[e + 1]]
        if rows.size == 0:
            continue
        tok = rows // k
        o[rows], u, v = _expert_rows(xq[tok], Wg[e], Wu[e], Wd[e], mx)
        if keep:
            u_all[rows], v_all[rows] = u, v
    y = np.zeros((T, d), f64)
    o_sh = None
    if n_shared:
        o_sh, _, _ = _expert_rows(xq, Wg[E], Wu[E], Wd[E], mx)
        y += o_sh
    for j in range(k):
        y += g[:, j:j + 1] * o[np.arange(T) * k + j]
    out = dict(r, y=y, o=o)
    if keep:
        out.update(u=u_all, v=v_all, o_shared=o_sh)
    return out


def _expert_rows(xr, Wg_e, Wu_e, Wd_e, mx: bool):
    if not mx:
        u, v, _, o = expert_ffn(xr, Wg_e, Wu_e, Wd_e)
        return o, u, v
    Wg_q = mx_fake_quant(Wg_e, axis=1)
    Wu_q = mx_fake_quant(Wu_e, axis=1)
    Wd_q = mx_fake_quant(Wd_e, axis=1)
    u = xr @ Wg_q.T
    v = xr @ Wu_q.T
    h = mx_fake_quant(silu(u) * v, axis=1)
    return h @ Wd_q.T, u, v


# --------------------------------------------------------------------------
# Backward
# --------------------------------------------------------------------------

def router_grad(logits, idx, g, dg, router: str, renorm: bool, scale: float):
    """dL/dlogits [T, E] from dL/dgate [T, k]. The selection bias gets no gradient.

    softmax, renorm:   dl_j = g_j (dg_j - sum_i g_i dg_i)          (selected experts only)
    softmax, all E:    dl_e = p_e (dg_e [e selected] - sum_j g_j dg_j)  (every expert)
    sigmoid, renorm:   dl_j = (scale/S)(dg_j - sum_i g_i dg_i / scale) s_j (1 - s_j),  S = sum_i s_i
    sigmoid, plain:    dl_j = scale dg_j s_j (1 - s_j)
    (a softmax router's scale multiplies dg first)
    """
    l = np.asarray(logits, f64)
    T, E = l.shape
    idx = np.asarray(idx).astype(np.int64)
    dl = np.zeros((T, E), f64)
    if router == "softmax":
        dgs = dg * scale
        gs = g / scale
        dot = np.sum(gs * dgs, axis=1, keepdims=True)
        if renorm:
            np.put_along_axis(dl, idx, gs * (dgs - dot), axis=1)
        else:
            m = l.max(axis=1, keepdims=True)
            p = np.exp(l - m)
            p = p / p.sum(axis=1, keepdims=True)
            dP = np.zeros((T, E), f64)
            np.put_along_axis(dP, idx, dgs, axis=1)
            dl = p * (dP - dot)
        return dl
    sel = np.take_along_axis(l, idx, axis=1)
    s = sigmoid(sel)
    if renorm:
        S = s.sum(axis=1, keepdims=True)
        ds = (scale / S) * (dg - np.sum(g * dg, axis=1, keepdims=True) / scale)
    else:
        ds = scale * dg
    np.put_along_axis(dl, idx, ds * s * (1.0 - s), axis=1)
    return dl


def mx_fake_quant_tokens(a):
    """MXFP8 values of a [n, ...] quantised along its token axis (axis 0) in blocks of 32 rows,
    the last block zero-padded (padding rows are dropped again)."""
    a = np.asarray(a, f64)
    n = a.shape[0]
    pad = (-n) % 32
    if pad:
        a = np.concatenate([a, np.zeros((pad,) + a.shape[1:], f64)])
    return mx_fake_quant(a, axis=0)[:n]


def backward(x, Wr, b, Wg, Wu, Wd, dy, k: int, router: str, renorm: bool, scale: float,
             n_shared: int = 0, logits32=None, mx: bool = False, experts=None):
    """Gradients of sum(y * dy) with respect to x, Wr, Wg, Wu, Wd (b gets none).

    Per assignment (expert e, token t, gate g):
      r = dy_t Wd[e]             dg = r . h          dh = g r
      du = dh v silu'(u)          dv = dh silu(u)
      dWd[e] += g dy_t^T h        dWg[e] += du^T x_t  dWu[e] += dv^T x_t
      dx_t += du Wg[e] + dv Wu[e]
    then the router: dl from dg, dWr = dl^T x, dx += dl Wr.

    mx=True: every expert GEMM operand is an MXFP8 value quantised along that
    GEMM's K (reading: E4M3 + E8M0 per 32 along K for activations and weights):
      forward   u, v from x (along d) and Wg, Wu (along d); h unquantised for dg
      r         dy (along d) times Wd (along d, i.e. its axis 0)
      dx        du, dv (along f) times Wg, Wu (along f, axis 0)
      dW        both operands along the expert's token axis (blocks of 32 tokens
                in sorted order, zero-padded): dWg = du^T x, dWu = dv^T x,
                dWd = dy^T (g h)
    The router GEMMs stay unquantised.

    experts (optional): evaluate only these experts (the shared expert is E);
    dWg, dWu, dWd are then dicts {expert: gradient} holding exactly those
    experts' gradients, while dx, dWr and dg miss the other experts' terms.
    Used to check single experts of a full-size layer.
    """
    x = np.asarray(x, f64)
    dy = np.asarray(dy, f64)
    if mx:
        xq = mx_fake_quant(x, axis=1)
        dyq = mx_fake_quant(dy, axis=1)
    T, d = x.shape
    E = np.asarray(Wr).shape[0]
    r = route(x, Wr, b, k, router, renorm, scale, logits32)
    idx, g, perm, off = r["idx"], r["gate"], r["perm"], r["off"]
    gflat = g.ravel()
    dx = np.zeros((T, d), f64)
    if experts is None:
        dWg = np.zeros(np.asarray(Wg).shape, f64)
        dWu = np.zeros(np.asarray(Wu).shape, f64)
        dWd = np.zeros(np.asarray(Wd).shape, f64)
    else:
        dWg, dWu, dWd = {}, {}, {}             # {expert: gradient} for the listed experts
    dg = np.zeros(T * k, f64)
    todo = [(e, perm[off[e]:off[e + 1]]) for e in range(E)]
    if n_shared:
        todo.append((E, None))
    if experts is not None:
        todo = [(e, rows) for e, rows in todo if e in set(experts)]
    for e, rows in todo:
        if rows is None:                      # shared expert: every token, gate 1
            tok = np.arange(T)
            ge = np.ones(T, f64)
        else:
            if rows.size == 0:
                continue
            tok = rows // k
            ge = gflat[rows]
        xr = x[tok]
        if not mx:
            u, v, h, _ = expert_ffn(xr, Wg[e], Wu[e], Wd[e])
            rr = dy[tok] @ np.asarray(Wd[e], f64)
        else:
            u = xq[tok] @ mx_fake_quant(Wg[e], axis=1).T
            v = xq[tok] @ mx_fake_quant(Wu[e], axis=1).T
            h = silu(u) * v
            rr = dyq[tok] @ mx_fake_quant(Wd[e], axis=0)
        if rows is not None:
            dg[rows] = np.sum(rr * h, axis=1)
        dh = ge[:, None] * rr
        du = dh * v * silu_grad(u)
        dv = dh * silu(u)
        if not mx:
            dWd[e] = (ge[:, None] * dy[tok]).T @ h
            dWg[e] = du.T @ xr
            dWu[e] = dv.T @ xr
            dx[tok] += du @ np.asarray(Wg[e], f64) + dv @ np.asarray(Wu[e], f64)
        else:
            xt = mx_fake_quant_tokens(xr)
            dWd[e] = mx_fake_quant_tokens(dy[tok]).T @ mx_fake_quant_tokens(ge[:, None] * h)
            dWg[e] = mx_fake_quant_tokens(du).T @ xt
            dWu[e] = mx_fake_quant_tokens(dv).T @ xt
            dx[tok] += (mx_fake_quant(du, axis=1) @ mx_fake_quant(Wg[e], axis=0) +
                        mx_fake_quant(dv, axis=1) @ mx_fake_quant(Wu[e], axis=0))
    dl = router_grad(r["logits"], idx, g, dg.reshape(T, k), router, renorm, scale)
    dWr = dl.T @ x
    dx += dl @ np.asarray(Wr, f64)
    return dict(r, dx=dx, dWr=dWr, dWg=dWg, dWu=dWu, dWd=dWd, dg=dg.reshape(T, k), dl=dl)


def loss(x, Wr, b, Wg, Wu, Wd, dy, **kw):
    """L = sum(y * dy): the scalar whose gradients backward() returns."""
    return float(np.sum(forward(x, Wr, b, Wg, Wu, Wd, **kw)["y"] * np.asarray(dy, f64)))


# --------------------------------------------------------------------------
# Chunked forward + backward over a fixed ring of saved activations
# [MoK, "Три решения ...": fixed ring buffer of a few hundred MB, walked in
#  reverse in the backward pass to reduce activation replay; 2368-token batches]
# --------------------------------------------------------------------------

def chunk_bounds(T: int, chunk: int):
    """[(t0, t1)] for consecutive chunks of `chunk` tokens; the last may be short."""
    if chunk <= 0 or chunk >= T:
        return [(0, T)]
    return [(t0, min(T, t0 + chunk)) for t0 in range(0, T, chunk)]


def ring_schedule(n_chunks: int, slots: int):
    """Events of a forward over chunks 0..n-1 then a backward over n-1..0 with `slots` ring slots.

    Forward chunk c saves into slot c mod slots. In the backward, chunk c finds
    its activations still resident iff no later chunk overwrote its slot, that is
    iff c >= n - slots; otherwise its forward is recomputed first.
    Returns a list of (phase, chunk, slot, recompute).
    """
    if slots < 1:
        raise ValueError("the ring needs at least one slot")
    ev = [("fwd", c, c % slots, False) for c in range(n_chunks)]
    for c in reversed(range(n_chunks)):
        ev.append(("bwd", c, c % slots, c < n_chunks - slots))
    return ev


def chunked_forward_backward(x, Wr, b, Wg, Wu, Wd, dy, chunk: int, **kw):
    """Forward and backward chunk by chunk; weight gradients summed over chunks in backward order.

    Tokens are independent in the layer, so this equals the unchunked result up
    to the order of the weight-gradient sums.
    """
    x = np.asarray(x, f64)
    bounds = chunk_bounds(x.shape[0], chunk)
    ys = [forward(x[a:b_], Wr, b, Wg, Wu, Wd, **kw)["y"] for a, b_ in bounds]
    dx = np.zeros_like(x)
    acc = None
    for a, b_ in reversed(bounds):
        g = backward(x[a:b_], Wr, b, Wg, Wu, Wd, np.asarray(dy, f64)[a:b_], **kw)
        dx[a:b_] = g["dx"]
        if acc is None:
            acc = {n: g[n].copy() for n in ("dWr", "dWg", "dWu", "dWd")}
        else:
            for n in acc:
                acc[n] += g[n]
    return dict(y=np.concatenate(ys), dx=dx, **acc)


# --------------------------------------------------------------------------
# Decode  [warp: small-batch decode; the same function as the forward at T = B]
# --------------------------------------------------------------------------

def decode(x, Wr, b, Wg, Wu, Wd, k, router, renorm, scale, n_shared=0, logits32=None, mx: bool = False):
    """Small-batch decode computes exactly the layer forward on B tokens (MXFP8 layers: the MXFP8 forward)."""
    return forward(x, Wr, b, Wg, Wu, Wd, k, router, renorm, scale, n_shared, logits32, mx=mx)


def rel_frobenius(a, ref):
    """||a - ref||_F / ||ref||_F."""
    a = np.asarray(a, f64)
    ref = np.asarray(ref, f64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))
