"""Plain float64 NumPy oracle for blockwise ring attention (test infrastructure).

Only tests, the smoke check and the bench's CPU-baseline leg use this module.
No blocking, fusion or reordering beyond what each docstring states.

Notation (the glossary page's toy uses the same names): N devices (blocks),
block = S / N tokens, dim = D.  q is [B, Hq, S, D]; k and v are [B, Hkv, S, D];
query head h reads key/value head h // (Hq // Hkv) (grouped-query attention,
the thienlv.com page's "compatible with GQA"; contiguous grouping is this
oracle's reading).  scale defaults to 1/sqrt(D) (the toy's ``dim**0.5``).

Layouts.  *Token order* is the sequence order.  *Shard-major* order is how N
devices hold the sequence: rows [i*Sb, (i+1)*Sb) belong to device i.  With the
contiguous layout shard-major equals token order; with the striped layout
(token t on device t mod N, the glossary page's Striped Attention remark, read
as round-robin assignment) row r of device i holds token r*N + i.
"""
from __future__ import annotations

import math

import numpy as np

FULL, INCL, STRICT = 0, 1, 2  # fold kinds: all pairs visible / u<=t diagonal / u<t diagonal


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact upcast of bfloat16 words (uint16) to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- layouts
CONTIGUOUS, STRIPED, ZIGZAG = 0, 1, 2


def positions(S: int, N: int, striped) -> np.ndarray:
    """Token position held by each shard-major row (length S, int64).

    Layouts (``striped`` is False/0, True/1 or 2):
      0 contiguous (aiunderstanding.org, "Immersione profonda": each device
        owns a contiguous block of tokens): row p holds token p;
      1 striped (glossary page, Striped Attention: tokens spread evenly over
        the devices, read as token t -> device t mod N, local row t div N):
        row i*Sb + r holds token r*N + i;
      2 zigzag (aiunderstanding.org page in Zulu, "Ikusasa": named as another
        causal load-balancing variant, not defined there; read as: cut the
        sequence into 2N chunks of Sb/2 tokens, device i holds chunk i then
        chunk 2N-1-i): row i*Sb + r holds token i*Sb/2 + r for r < Sb/2 and
        (2N-1-i)*Sb/2 + (r - Sb/2) otherwise.
    """
    if S % N:
        raise ValueError("S must be a multiple of N")
    Sb = S // N
    p = np.arange(S, dtype=np.int64)
    layout = int(striped)
    if layout == CONTIGUOUS:
        return p
    i, r = p // Sb, p % Sb
    if layout == STRIPED:
        return r * N + i
    if layout == ZIGZAG:
        if Sb % 2:
            raise ValueError("zigzag needs an even shard size")
        h = Sb // 2
        return np.where(r < h, i * h + r, (2 * N - 1 - i) * h + (r - h))
    raise ValueError(f"unknown layout {striped}")


def stripe_perm(S: int, N: int, layout=1) -> np.ndarray:
    """perm[p] = token held by shard-major row p (striped layout by default)."""
    return positions(S, N, layout)


def to_shard_major(x_tok: np.ndarray, N: int, striped: bool) -> np.ndarray:
    """Token order -> shard-major order along axis -2."""
    return x_tok[..., positions(x_tok.shape[-2], N, striped), :]


def to_token_order(x_sm: np.ndarray, N: int, striped: bool) -> np.ndarray:
    """Shard-major order -> token order along axis -2 (inverse of to_shard_major)."""
    pos = positions(x_sm.shape[-2], N, striped)
    out = np.empty_like(x_sm)
    out[..., pos, :] = x_sm
    return out


def _scale(D: int, scale) -> float:
    return 1.0 / math.sqrt(D) if scale is None or scale <= 0 else float(scale)


# ------------------------------------------------------- plain definition
def attend_rows(qrows, qpos, k, v, kpos, causal: bool, scale: float):
    """Exact softmax attention for a set of query rows (the plain definition).

    For each query row t with position qpos[t], keys u with kpos[u] <= qpos[t]
    are visible when ``causal`` (standard inclusive causal mask; the pages do
    not state the convention, this is the oracle's reading), all keys
    otherwise.  Returns
        O[t]   = sum_u softmax_u(scale * q_t . k_u) v_u
        lse[t] = ln sum_u exp(scale * q_t . k_u)
    computed with the maximum subtracted before exp (the glossary page notes
    production kernels do so; it changes nothing mathematically).  A row with
    no visible key gets O = 0, lse = -inf.
    """
    qrows = np.asarray(qrows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (qrows @ k.T) * scale  # [R, Sk]
    if causal:
        vis = np.asarray(kpos)[None, :] <= np.asarray(qpos)[:, None]
        s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe)
    l = p.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l > 0, (p @ v) / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[:, 0] > 0, m_safe[:, 0] + np.log(l[:, 0]), -np.inf)
    return o, lse


def full_attention(q, k, v, causal: bool, scale=None, chunk: int = 512):
    """Full softmax(scale * Q K^T) V over token-order tensors, float64.

    q [B, Hq, S, D], k and v [B, Hkv, S, D].  Query rows are processed in
    chunks of ``chunk`` rows only to bound memory; each chunk is the plain
    definition (``attend_rows``).  Returns O [B, Hq, S, D], lse [B, Hq, S].
    """
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    sc = _scale(D, scale)
    o = np.empty((B, Hq, S, v.shape[-1]), dtype=np.float64)
    lse = np.empty((B, Hq, S), dtype=np.float64)
    pos = np.arange(S, dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            for r0 in range(0, S, chunk):
                r1 = min(S, r0 + chunk)
                hi = r1 if causal else S  # keys beyond the last row are invisible
                o[b, h, r0:r1], lse[b, h, r0:r1] = attend_rows(
                    q[b, h, r0:r1], pos[r0:r1], kh[:hi], vh[:hi], pos[:hi], causal, sc)
    return o, lse


# ------------------------------------------------------- ring-order loop
def ring_attention(q, k, v, N: int, causal: bool, striped: bool, scale=None):
    """Blockwise ring attention over shard-major tensors, float64.

    Follows the glossary page ("Como funciona a atencao em anel") and the
    aiunderstanding.org "Approfondimento tecnico" section: device i keeps
    query block Q_i; at step s = 0..N-1 it holds key/value block
    j = (i - s) mod N (received from the previous device, so step 0 is its
    own block).  For each block it forms the scores scale * Q_i K_j^T, masks
    pairs whose key position is after the query position (causal), and folds
    them into a running max m, running normaliser l and numerator acc:
        m'  = max(m, rowmax(scores))
        acc = exp(m - m') * acc + exp(scores - m') @ V_j
        l   = exp(m - m') * l   + rowsum(exp(scores - m'))
    (with exp(m - m') taken as 0 while m = -inf).  Blocks with no visible
    pair are skipped.  After the N steps O_i = acc / l and lse = m + ln l.
    Returns O and lse in shard-major order.
    """
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    Sb = S // N
    sc = _scale(D, scale)
    pos = positions(S, N, striped)
    o = np.zeros((B, Hq, S, v.shape[-1]), dtype=np.float64)
    lse = np.full((B, Hq, S), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            Q = np.asarray(q[b, h], dtype=np.float64)
            K = np.asarray(k[b, h // g], dtype=np.float64)
            V = np.asarray(v[b, h // g], dtype=np.float64)
            for i in range(N):
                qi = slice(i * Sb, (i + 1) * Sb)
                m = np.full(Sb, -np.inf)
                l = np.zeros(Sb)
                acc = np.zeros((Sb, V.shape[1]))
                for s in range(N):
                    j = (i - s) % N
                    kj = slice(j * Sb, (j + 1) * Sb)
                    scores = (Q[qi] @ K[kj].T) * sc
                    if causal:
                        vis = pos[kj][None, :] <= pos[qi][:, None]
                        if not vis.any():
                            continue
                        scores = np.where(vis, scores, -np.inf)
                    m_new = np.maximum(m, scores.max(axis=1))
                    m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)
                    p = np.exp(scores - m_use[:, None])
                    acc = alpha[:, None] * acc + p @ V[kj]
                    l = alpha * l + p.sum(axis=1)
                    m = m_new
                with np.errstate(invalid="ignore", divide="ignore"):
                    o[b, h, qi] = np.where(l[:, None] > 0, acc / np.where(l > 0, l, 1)[:, None], 0)
                    lse[b, h, qi] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1)), -np.inf)
    return o, lse


def merge(o_a, lse_a, o_b, lse_b):
    """Combine two partial results over disjoint key sets A and B.

    With lse_X = ln sum_{u in X} exp(score_u) and O_X the normalised partial
    output, the result over A u B is the log-sum-exp weighting (the same
    rescale-and-add the pages' online softmax performs when a block arrives):
        lse = ln(exp(lse_a) + exp(lse_b))
        O   = exp(lse_a - lse) O_a + exp(lse_b - lse) O_b
    A partial over no visible key has lse = -inf and contributes nothing; if
    both are empty the result is O = 0, lse = -inf.
    """
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    mx = np.maximum(lse_a, lse_b)
    mx_safe = np.where(np.isfinite(mx), mx, 0.0)
    wa = np.exp(lse_a - mx_safe)
    wb = np.exp(lse_b - mx_safe)
    tot = wa + wb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, mx_safe + np.log(np.where(tot > 0, tot, 1)), -np.inf)
        ca = np.where(tot > 0, wa / np.where(tot > 0, tot, 1), 0.0)
        cb = np.where(tot > 0, wb / np.where(tot > 0, tot, 1), 0.0)
    o = ca[..., None] * np.asarray(o_a, np.float64) + cb[..., None] * np.asarray(o_b, np.float64)
    return o, lse


# ------------------------------------------------------------- gradients
def attention_backward(q, k, v, dout, causal: bool, scale=None, chunk: int = 512):
    """Gradients of the plain definition with respect to q, k and v, float64.

    The pages use the method to train long-context models (the Italian
    aiunderstanding.org page, "Implementazione nel mondo reale": training an
    LLM on 1M-token sequences; the glossary page: end-to-end training
    throughput, and PyTorch's context_parallel replacing scaled dot-product
    attention in training).  They do not write the backward out, so this is
    the chain rule applied to O = softmax(scale Q K^T) V, row by row, with
    dO = dL/dO given.  For query row t and its visible keys u:
        P_tu  = softmax_u(scale q_t . k_u)
        dV_u  = sum_t P_tu dO_t
        dP_tu = dO_t . v_u
        dS_tu = P_tu (dP_tu - sum_u' P_tu' dP_tu')      (softmax Jacobian)
        dQ_t  = scale sum_u dS_tu k_u
        dK_u  = scale sum_t dS_tu q_t
    With grouped-query attention a key/value head's gradient is the sum over
    the query heads that read it.  Token-order tensors; query rows are taken
    in chunks of ``chunk`` only to bound memory.  Returns dq, dk, dv.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    sc = _scale(D, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pos = np.arange(S, dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            for r0 in range(0, S, chunk):
                r1 = min(S, r0 + chunk)
                s = (q[b, h, r0:r1] @ kh.T) * sc
                if causal:
                    s = np.where(pos[None, :] <= pos[r0:r1, None], s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                m = np.where(np.isfinite(m), m, 0.0)
                e = np.exp(s - m)
                den = e.sum(axis=1, keepdims=True)
                P = e / np.where(den > 0, den, 1.0)
                dP = dout[b, h, r0:r1] @ vh.T
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dv[b, h // g] += P.T @ dout[b, h, r0:r1]
                dq[b, h, r0:r1] = sc * (dS @ kh)
                dk[b, h // g] += sc * (dS.T @ q[b, h, r0:r1])
    return dq, dk, dv


def attention_backward_rows(qrows, qpos, dorows, k, v, kpos, causal: bool, scale: float):
    """dq for a set of query rows of one head, from the plain definition.

    For each query row t (position qpos[t], dL/dout row dorows[t]) against
    the keys k, v of its key/value head (positions kpos): P_t = softmax of
    the visible scores, dP_tu = dO_t . v_u, dS_tu = P_tu (dP_tu - sum_u'
    P_tu' dP_tu'), dq_t = scale sum_u dS_tu k_u -- the rows of
    ``attention_backward``'s dq, for rows chosen by the caller.
    """
    qrows = np.asarray(qrows, np.float64)
    dorows = np.asarray(dorows, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = (qrows @ k.T) * scale
    if causal:
        s = np.where(np.asarray(kpos)[None, :] <= np.asarray(qpos)[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m)
    den = e.sum(axis=1, keepdims=True)
    P = e / np.where(den > 0, den, 1.0)
    dP = dorows @ v.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    return scale * (dS @ k)


def attention_backward_key_rows(qrows, qpos, dorows, k, v, kpos, keys, causal: bool,
                                scale: float, chunk: int = 256):
    """dk and dv of chosen key rows of one head, from the plain definition.

    qrows [T, D] with positions qpos and dL/dout rows dorows [T, D] must hold
    every query row that sees any chosen key (under the causal mask, every
    query at or after the earliest chosen key's position); k, v [Sk, D] are
    all keys and values of the head with positions kpos; ``keys`` indexes the
    chosen rows of k.  For each query row t (taken ``chunk`` rows at a time
    only to bound memory), over its visible keys u:
        P_tu  = softmax_u(scale q_t . k_u)
        dP_tu = dO_t . v_u
        dS_tu = P_tu (dP_tu - sum_u' P_tu' dP_tu')     (softmax Jacobian)
    and for each chosen key c
        dK_c = scale sum_t dS_tc q_t,    dV_c = sum_t P_tc dO_t
    -- the rows ``keys`` of ``attention_backward``'s dk and dv for one query
    head (a key/value head's gradient is the sum over its query heads).
    Returns dk [len(keys), D], dv [len(keys), D].
    """
    qrows = np.asarray(qrows, np.float64)
    dorows = np.asarray(dorows, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    qpos = np.asarray(qpos)
    kpos = np.asarray(kpos)
    keys = np.asarray(keys, np.int64)
    dk = np.zeros((len(keys), k.shape[1]))
    dv = np.zeros((len(keys), v.shape[1]))
    for r0 in range(0, len(qrows), chunk):
        q, do, qp = qrows[r0:r0 + chunk], dorows[r0:r0 + chunk], qpos[r0:r0 + chunk]
        s = (q @ k.T) * scale
        if causal:
            s = np.where(kpos[None, :] <= qp[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        P = e / np.where(den > 0, den, 1.0)
        dP = do @ v.T
        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dk += scale * (dS[:, keys].T @ q)
        dv += P[:, keys].T @ do
    return dk, dv


def backward_uniform_scores(q, v, dout, causal: bool, scale=None, dk_rows=None):
    """dk and dv of the plain definition when every score is zero (K = 0),
    token order, float64, by prefix sums.

    Every query row t then weighs its n_t visible keys equally (n_t = t + 1
    under the causal mask, S otherwise), and the definition reduces to
        dv_u = sum over rows t that see u of dO_t / n_t
        m_t  = dO_t . (mean of the v_u row t sees)          (= sum_u P_tu dP_tu)
        dk_u = scale sum over rows t that see u of (dO_t . v_u - m_t) q_t / n_t
    (dq is zero, as every k_u is).  A key/value head's gradients sum over the
    query heads that read it.  q [B, Hq, S, D], v [B, Hkv, S, D], dout like q.
    Returns dv [B, Hkv, S, D] and dk for the key positions in ``dk_rows``
    ([B, Hkv, len(dk_rows), D]; all rows when None).
    """
    q = np.asarray(q, np.float64)
    v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    B, Hq, S, D = q.shape
    Hkv = v.shape[1]
    g = Hq // Hkv
    sc = _scale(D, scale)
    rows = np.arange(S) if dk_rows is None else np.asarray(dk_rows, np.int64)
    n = np.arange(1, S + 1, dtype=np.float64) if causal else np.full(S, float(S))
    dv = np.zeros((B, Hkv, S, D))
    dk = np.zeros((B, Hkv, len(rows), D))
    for b in range(B):
        for h in range(Hq):
            V, dO, Q = v[b, h // g], dout[b, h], q[b, h]
            w = dO / n[:, None]
            if causal:
                dv[b, h // g] += np.cumsum(w[::-1], axis=0)[::-1]    # sum over t >= u
                vbar = np.cumsum(V, axis=0) / n[:, None]             # mean of v_0..v_t
            else:
                dv[b, h // g] += w.sum(axis=0)[None, :]
                vbar = np.broadcast_to(V.mean(axis=0), V.shape)
            m = (dO * vbar).sum(axis=1)
            for e, u in enumerate(rows):
                t0 = u if causal else 0
                c = (dO[t0:] @ V[u] - m[t0:]) / n[t0:]
                dk[b, h // g, e] += sc * (c @ Q[t0:])
    return dk, dv


def ring_attention_backward(q, k, v, dout, N: int, causal: bool, striped, scale=None):
    """Backward of ``ring_attention`` folded in ring order, float64.

    Reading (the pages name training as the use but leave the backward
    open): the same ring as the forward, with each key/value block carrying
    its gradient accumulators dK_j, dV_j as it travels, while dQ_i stays on
    device i.  Before the ring each device has the forward's lse_i and O_i
    and forms delta_t = dO_t . O_t, which equals sum_u P_tu dP_tu.  At step
    s = 0..N-1 device i holds block j = (i - s) mod N and, for the visible
    pairs of Q_i and K_j (other pairs have P = 0; a block with none is
    skipped):
        P     = exp(scale Q_i K_j^T - lse_i)
        dV_j += P^T dO_i
        dP    = dO_i V_j^T
        dS    = P * (dP - delta_i)
        dQ_i += scale dS K_j
        dK_j += scale dS^T Q_i
    Shard-major tensors in, shard-major gradients out.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dout = np.asarray(dout, np.float64)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    Sb = S // N
    sc = _scale(D, scale)
    pos = positions(S, N, striped)
    o, lse = ring_attention(q, k, v, N, causal, striped, scale)
    delta = (dout * o).sum(axis=-1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            Q, dO = q[b, h], dout[b, h]
            K, V = k[b, h // g], v[b, h // g]
            dK, dV = dk[b, h // g], dv[b, h // g]
            for s in range(N):
                for i in range(N):
                    j = (i - s) % N
                    qi = slice(i * Sb, (i + 1) * Sb)
                    kj = slice(j * Sb, (j + 1) * Sb)
                    vis = (pos[kj][None, :] <= pos[qi][:, None]) if causal else \
                        np.ones((Sb, Sb), dtype=bool)
                    if not vis.any():
                        continue
                    with np.errstate(invalid="ignore"):
                        P = np.where(vis, np.exp((Q[qi] @ K[kj].T) * sc - lse[b, h, qi][:, None]),
                                     0.0)
                    dV[kj] += P.T @ dO[qi]
                    dP = dO[qi] @ V[kj].T
                    dS = P * (dP - delta[b, h, qi][:, None])
                    dq[b, h, qi] += sc * (dS @ K[kj])
                    dK[kj] += sc * (dS.T @ Q[qi])
    return dq, dk, dv


def ring_step_backward_block(q_i, k_j, v_j, dout_i, lse_i, delta_i, N: int, i: int, j: int,
                             causal: bool, striped, scale=None):
    """One step of ``ring_attention_backward`` as a device computes it,
    float64: device i's query shard (q_i, dout_i [B, Hq, Sb, D], its forward
    lse_i and delta_i = dO_t . O_t [B, Hq, Sb]) against the block j it holds
    (k_j, v_j [B, Hkv, Sb, D]).  Returns (dq_i, dk_j, dv_j): the terms this
    step adds to the shard's dq and to the block's travelling dk and dv, by
    the same formulas (P = exp(scale q.k - lse) on the visible pairs, dS =
    P (dO.v - delta)).  Summed over the ring's steps they give the whole
    backward.
    """
    q_i = np.asarray(q_i, np.float64)
    k_j = np.asarray(k_j, np.float64)
    v_j = np.asarray(v_j, np.float64)
    dout_i = np.asarray(dout_i, np.float64)
    lse_i = np.asarray(lse_i, np.float64)
    delta_i = np.asarray(delta_i, np.float64)
    B, Hq, Sb, D = q_i.shape
    Hkv = k_j.shape[1]
    g = Hq // Hkv
    sc = _scale(D, scale)
    pos = positions(N * Sb, N, striped)
    qpos, kpos = pos[i * Sb:(i + 1) * Sb], pos[j * Sb:(j + 1) * Sb]
    vis = (kpos[None, :] <= qpos[:, None]) if causal else np.ones((Sb, Sb), dtype=bool)
    dq = np.zeros_like(q_i)
    dk = np.zeros_like(k_j)
    dv = np.zeros_like(v_j)
    if not vis.any():
        return dq, dk, dv
    for b in range(B):
        for h in range(Hq):
            Q, dO = q_i[b, h], dout_i[b, h]
            K, V = k_j[b, h // g], v_j[b, h // g]
            with np.errstate(invalid="ignore", over="ignore"):
                P = np.where(vis, np.exp((Q @ K.T) * sc - lse_i[b, h][:, None]), 0.0)
            dv[b, h // g] += P.T @ dO
            dS = P * (dO @ V.T - delta_i[b, h][:, None])
            dq[b, h] = sc * (dS @ K)
            dk[b, h // g] += sc * (dS.T @ Q)
    return dq, dk, dv


# ------------------------------------------------------------- schedule
def fold_schedule(S: int, N: int, causal: bool, striped: bool, Tq: int, Tk: int,
                  i_list=None, qt_list=None):
    """Brute-force fold order of every query tile, from explicit positions.

    For query shard i, query tile qt (rows [qt*Tq, (qt+1)*Tq) of the shard)
    and ring step s = 0..N-1 with j = (i - s) mod N, walk the key tiles kt of
    shard j in ascending order and classify the Tq x Tk pairs from their
    token positions: no visible pair -> skipped (not listed); all visible ->
    FULL; exactly the pairs with local key row <= local query row -> INCL;
    exactly those with local key row < local query row -> STRICT.  Any other
    pattern raises (the tile sizes do not fit the layout).

    Returns a list of (i, qt, s, j, kt, kind) in fold order.
    """
    Sb = S // N
    pos = positions(S, N, striped)
    nq, nk = -(-Sb // Tq), -(-Sb // Tk)
    out = []
    for i in (range(N) if i_list is None else i_list):
        for qt in (range(nq) if qt_list is None else qt_list):
            r0, r1 = i * Sb + qt * Tq, i * Sb + min(Sb, (qt + 1) * Tq)
            rl = np.arange(r1 - r0)
            for s in range(N):
                j = (i - s) % N
                for kt in range(nk):
                    c0, c1 = j * Sb + kt * Tk, j * Sb + min(Sb, (kt + 1) * Tk)
                    cl = np.arange(c1 - c0)
                    if causal:
                        vis = pos[c0:c1][None, :] <= pos[r0:r1][:, None]
                    else:
                        vis = np.ones((r1 - r0, c1 - c0), dtype=bool)
                    if not vis.any():
                        continue
                    if vis.all():
                        kind = FULL
                    elif (r1 - r0 == c1 - c0) and np.array_equal(vis, cl[None, :] <= rl[:, None]):
                        kind = INCL
                    elif (r1 - r0 == c1 - c0) and np.array_equal(vis, cl[None, :] < rl[:, None]):
                        kind = STRICT
                    else:
                        raise ValueError(f"unclassifiable tile i={i} qt={qt} j={j} kt={kt}")
                    out.append((i, qt, s, j, kt, kind))
    return out


# ------------------------------------------------- head/sequence exchange
def ulysses_exchange(x, N: int, inverse: bool = False):
    """The all-to-all of DeepSpeed Ulysses as a permutation between N
    device-contiguous buffers (glossary page, "Atencao em anel vs. outros
    tipos de paralelismo": the exchange gives each device every token of a
    subset of the attention heads).

    Forward: x is sequence-sharded [N, B, H, S/N, ...] (device i holds tokens
    [i*S/N, (i+1)*S/N) of every head); the result is head-sharded
    [N, B, H/N, S, ...] (device d holds heads [d*H/N, (d+1)*H/N), every token
    in order):  out[d, b, hl, t] = x[t // (S/N), b, d*H/N + hl, t % (S/N)].
    inverse=True maps back.  H must be a multiple of N.
    """
    x = np.asarray(x)
    if not inverse:
        n, B, H, Sb = x.shape[:4]
        if n != N or H % N:
            raise ValueError("bad shapes")
        Hl, S = H // N, N * Sb
        out = np.empty((N, B, Hl, S) + x.shape[4:], dtype=x.dtype)
        for d in range(N):
            for hl in range(Hl):
                for t in range(S):
                    out[d, :, hl, t] = x[t // Sb, :, d * Hl + hl, t % Sb]
        return out
    n, B, Hl, S = x.shape[:4]
    if n != N or S % N:
        raise ValueError("bad shapes")
    Sb, H = S // N, N * Hl
    out = np.empty((N, B, H, Sb) + x.shape[4:], dtype=x.dtype)
    for i in range(N):
        for h in range(H):
            for r in range(Sb):
                out[i, :, h, r] = x[h // Hl, :, h % Hl, i * Sb + r]
    return out


# ----------------------------------------------------- the pages' toy
def toy_ring_no_max(q, k, v, n_devices: int):
    """The glossary page's four-device simulation, as its text describes it.

    q, k, v are [n_devices * block, dim] in token order.  Device i keeps its
    query block; at each step it takes the key/value block j = (i - step) mod
    n_devices, adds exp(Q_i K_j^T / sqrt(dim)) @ V_j to a numerator and the
    row sums of exp(...) to a denominator, and finally divides.  No running
    maximum is subtracted (the page's simulation omits it).  float64.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    S, dim = q.shape
    blk = S // n_devices
    outs = []
    for i in range(n_devices):
        num = np.zeros((blk, v.shape[1]))
        den = np.zeros((blk, 1))
        Qi = q[i * blk:(i + 1) * blk]
        for step in range(n_devices):
            j = (i - step) % n_devices
            e = np.exp(Qi @ k[j * blk:(j + 1) * blk].T / math.sqrt(dim))
            num += e @ v[j * blk:(j + 1) * blk]
            den += e.sum(axis=1, keepdims=True)
        outs.append(num / den)
    return np.concatenate(outs, axis=0)
