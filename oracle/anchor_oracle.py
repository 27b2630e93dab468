"""fp64 CPU oracle for fused RoPE + AnchorAttention (forward and backward).

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs use it. It shares no code with the CUDA library: it builds the
explicit mask and the position IDs from their definitions and evaluates the
attention densely, in float64, with numpy.

Sources (all from the web pages on arXiv 2411.13476, "When Precision Meets
Position: BFloat16 Breaks Down RoPE in Long-Context Training"):

* RoPE rotation, Eq. 6 (architecture page, §3.4 "Rotary Positional Embedding
  (RoPE): The Theoretical Promise"): block-diagonal 2x2 rotations of the
  adjacent coordinate pairs (2p, 2p+1) by the angle i*theta_p with
  theta_p = base^(-2p/d), p = 0 .. d/2-1.
* Attention with a mask (same section, "Standard attention"): masked logits,
  softmax over the attended positions, weighted sum of values. The 1/sqrt(d)
  scale that the page omits "for simplicity" is restored as ``softmax_scale``.
* AnchorAttention mask (architecture page, §3.4 "AnchorAttention: The Shared
  Anchor Design", "Mask construction"): every token sees the anchor (column
  0); intra-document causal j <= i; cross-document and future positions are
  masked; the anchor itself sees only itself.
* Position IDs (architecture page, §3.4 "Document Token Indexing"):
  continuous IDs (Fig. 2 left), IDs reset to 1 at every document start
  (Fig. 2 middle); the anchor sits at position 0 (§3.4 "AnchorAttention",
  "Core design", item 1).

Readings where the pages are silent or disagree (each is also listed in the
design notes): the default position scheme is RESET (every document restarts
at 1, the anchor alone is at 0); CONTINUOUS is the pages' own "Core design"
item 2 and is supported equally. INTRA_DOC mode makes the anchor token its own
one-token document. LSE is the natural-log logsumexp of the scaled logits.
The backward pass is the analytic gradient of this forward with respect to the
un-rotated q, k and v (so it includes the transposed rotation R^T).

Parity status: every function here is pinned by ``tests/test_oracle.py``
against hand-enumerated masks, closed forms, an independent library
attention, complex-number rotation and finite differences.
"""
from __future__ import annotations

import numpy as np

# Enumerations: the numeric values are part of the library's interface.
MASK_CAUSAL, MASK_INTRA_DOC, MASK_ANCHOR = 0, 1, 2
POS_RESET, POS_CONTINUOUS = 0, 1
ROPE_ADJACENT, ROPE_HALF, ROPE_NONE = 0, 1, 2


def _check_cu(cu_doclens, T):
    cu = np.asarray(cu_doclens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_doclens needs at least one document")
    if cu[0] != 1 or cu[-1] != T or np.any(np.diff(cu) <= 0):
        raise ValueError("cu_doclens must start at 1, end at T and increase strictly")
    return cu


def document_ids(cu_doclens, T: int, mask_mode: int) -> np.ndarray:
    """Document index of each token: anchor = 0, documents 1..K.

    In CAUSAL mode the whole packed sequence is one sequence (all zeros) and
    cu_doclens is not consulted.
    """
    doc = np.zeros(T, dtype=np.int64)
    if mask_mode == MASK_CAUSAL:
        return doc
    cu = _check_cu(cu_doclens, T)
    for k in range(1, cu.size):
        doc[cu[k - 1]:cu[k]] = k
    return doc


def position_ids(cu_doclens, T: int, mask_mode: int, pos_mode: int,
                 pos_shift: int = 0) -> np.ndarray:
    """Rotation index of each token (the i of R_{i,theta}).

    CONTINUOUS (and CAUSAL): 0, 1, 2, ... T-1 over the packed sequence.
    RESET: the anchor is 0; the tokens of every document are 1, 2, ..., N_k.
    ``pos_shift`` adds the same Delta to every position (Eq. 3 diagnostics).
    """
    if mask_mode == MASK_CAUSAL or pos_mode == POS_CONTINUOUS:
        pos = np.arange(T, dtype=np.int64)
    elif pos_mode == POS_RESET:
        cu = _check_cu(cu_doclens, T)
        pos = np.zeros(T, dtype=np.int64)
        for k in range(1, cu.size):
            n = cu[k] - cu[k - 1]
            pos[cu[k - 1]:cu[k]] = np.arange(1, n + 1)
    else:
        raise ValueError("unknown position mode")
    return pos + int(pos_shift)


def segment_position_ids(doc_of_token, pos_mode: int, pos_shift: int = 0) -> np.ndarray:
    """Positions for documents given per token (interleaved chunks).

    Architecture page, §3.4 "AnchorAttention with Interleaved Chunks": chunks
    of one document keep their order, so a document's tokens are its tokens
    in sequence order. RESET ("Document Token Indexing", Fig. 2 middle)
    counts 1, 2, ... through them; CONTINUOUS is the token index; the anchor
    (token 0) is at 0. ``pos_shift`` adds to every position (Eq. 3).
    """
    doc = np.asarray(doc_of_token, dtype=np.int64)
    T = doc.size
    if pos_mode == POS_CONTINUOUS:
        return np.arange(T, dtype=np.int64) + pos_shift
    pos = np.zeros(T, dtype=np.int64)
    seen = {}
    for i in range(1, T):
        seen[doc[i]] = seen.get(doc[i], 0) + 1
        pos[i] = seen[doc[i]]
    return pos + pos_shift


def mask_rows(rows, doc: np.ndarray, mask_mode: int) -> np.ndarray:
    """Boolean "may attend" matrix for the given query rows against all keys.

    The four rules of "Mask construction" (ANCHOR); INTRA_DOC drops the anchor
    exception; CAUSAL keeps only j <= i.
    """
    rows = np.asarray(rows, dtype=np.int64)
    T = doc.size
    j = np.arange(T, dtype=np.int64)[None, :]
    i = rows[:, None]
    causal = j <= i                                   # M = -inf if j > i
    if mask_mode == MASK_CAUSAL:
        return causal
    same_doc = doc[rows][:, None] == doc[None, :]     # -inf across documents
    allowed = causal & same_doc                       # intra-document causal
    if mask_mode == MASK_ANCHOR:
        allowed[:, 0] = True                          # M_{i,0} = 0 for all i
    elif mask_mode != MASK_INTRA_DOC:
        raise ValueError("unknown mask mode")
    return allowed


def attention_mask(cu_doclens, T: int, mask_mode: int) -> np.ndarray:
    """The explicit T x T mask (True = visible)."""
    doc = document_ids(cu_doclens, T, mask_mode)
    return mask_rows(np.arange(T), doc, mask_mode)


def unmasked_pairs(cu_doclens, T: int, mask_mode: int, block: int = 2048) -> int:
    """Number of visible (query, key) pairs, counted from the explicit mask."""
    doc = document_ids(cu_doclens, T, mask_mode)
    total = 0
    for r0 in range(0, T, block):
        total += int(mask_rows(np.arange(r0, min(T, r0 + block)), doc, mask_mode).sum())
    return total


def tile_counts(cu_doclens, T: int, mask_mode: int, tile: int = 128):
    """(live, causal) numbers of tile x tile blocks of the explicit mask.

    live: blocks holding at least one visible pair; causal: blocks holding at
    least one pair with j <= i (what full causal attention would visit).
    """
    doc = document_ids(cu_doclens, T, mask_mode)
    nt = (T + tile - 1) // tile
    live = 0
    for a in range(nt):
        m = mask_rows(np.arange(a * tile, min(T, (a + 1) * tile)), doc, mask_mode)
        for b in range(a + 1):
            if m[:, b * tile:min(T, (b + 1) * tile)].any():
                live += 1
    return live, nt * (nt + 1) // 2


def rope_theta(d: int, base: float) -> np.ndarray:
    """theta_p = base^(-2p/d), p = 0 .. d/2-1 (Eq. 6), in float64."""
    p = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * p / d)


def rotate(x, pos, base: float, layout: int = ROPE_ADJACENT, inverse: bool = False, theta=None):
    """Apply R_{pos,theta} (or its transpose) to x [T, H, d]; float64 out.

    ADJACENT pairs coordinates (2p, 2p+1) exactly as Eq. 6; HALF pairs
    (p, p + d/2); NONE returns x unchanged. Angles are pos * theta_p in fp64,
    theta_p = base^(-2p/d) unless an explicit table ``theta`` [d/2] is given
    (a RoPE variant's frequencies: Eq. 6 with other theta_p).
    """
    x = np.asarray(x, dtype=np.float64)
    if layout == ROPE_NONE:
        return x.copy()
    T, H, d = x.shape
    theta = rope_theta(d, base) if theta is None else np.asarray(theta, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]   # [T, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if inverse:
        s = -s
    if layout == ROPE_ADJACENT:
        a, b = x[..., 0::2], x[..., 1::2]
    elif layout == ROPE_HALF:
        a, b = x[..., : d // 2], x[..., d // 2:]
    else:
        raise ValueError("unknown rope layout")
    ra = c * a - s * b
    rb = s * a + c * b
    out = np.empty_like(x)
    if layout == ROPE_ADJACENT:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


class Problem:
    """One packed-attention problem: shapes, mask mode, positions and RoPE."""

    def __init__(self, cu_doclens, T, num_q_heads, num_kv_heads, head_dim,
                 rope_base=1e4, mask_mode=MASK_ANCHOR, pos_mode=POS_RESET,
                 rope_layout=ROPE_ADJACENT, softmax_scale=None, pos_shift=0, theta=None, doc_of_token=None):
        if num_q_heads % num_kv_heads:
            raise ValueError("query heads must be a multiple of kv heads")
        self.T, self.Hq, self.Hkv, self.d = T, num_q_heads, num_kv_heads, head_dim
        self.base, self.mask_mode, self.pos_mode = rope_base, mask_mode, pos_mode
        self.layout = rope_layout
        self.scale = (1.0 / np.sqrt(head_dim)) if not softmax_scale or softmax_scale <= 0 \
            else float(softmax_scale)
        if doc_of_token is not None:
            # documents given per token: token 0 is the anchor (0), the rest name
            # their document (>= 1); the mask compares these ids directly
            doc = np.asarray(doc_of_token, dtype=np.int64)
            if doc.shape != (T,) or doc[0] != 0 or np.any(doc[1:] < 1) or mask_mode == MASK_CAUSAL:
                raise ValueError("doc_of_token: [T] ids, 0 for the anchor only, ANCHOR or INTRA_DOC mode")
            self.cu = None
            self.doc = doc
            self.pos = segment_position_ids(doc, pos_mode, pos_shift)
        else:
            self.cu = None if mask_mode == MASK_CAUSAL else _check_cu(cu_doclens, T)
            self.doc = document_ids(cu_doclens, T, mask_mode)
            self.pos = position_ids(cu_doclens, T, mask_mode, pos_mode, pos_shift)
        self.theta = None if theta is None else np.asarray(theta, dtype=np.float64)

    def kv_head(self, h):
        """Grouped-query mapping: query head h reads kv head floor(h * Hkv / Hq)."""
        return (h * self.Hkv) // self.Hq

    def rotated(self, q, k):
        qr = rotate(np.asarray(q, np.float64), self.pos, self.base, self.layout, theta=self.theta)
        kr = rotate(np.asarray(k, np.float64), self.pos, self.base, self.layout, theta=self.theta)
        return qr, kr


def _as64(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def forward(prob: Problem, q, k, v, rows=None):
    """O [len(rows), Hq, d] and LSE [Hq, len(rows)] for the given query rows.

    s_ij = scale * (R_i q_i) . (R_j k_j) on visible pairs; P = softmax_j(s);
    O_i = sum_j P_ij v_j; LSE_i = ln sum_j exp(s_ij).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    rows = np.arange(prob.T) if rows is None else np.asarray(rows, dtype=np.int64)
    qr, kr = prob.rotated(q, k)
    allowed = mask_rows(rows, prob.doc, prob.mask_mode)
    O = np.zeros((rows.size, prob.Hq, prob.d))
    L = np.zeros((prob.Hq, rows.size))
    for h in range(prob.Hq):
        g = prob.kv_head(h)
        s = prob.scale * (qr[rows, h, :] @ kr[:, g, :].T)
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        P = e / z
        O[:, h, :] = P @ v[:, g, :]
        L[h, :] = (m + np.log(z))[:, 0]
    return O, L


def backward(prob: Problem, q, k, v, dout, rows=None):
    """Gradients (dq, dk, dv) of sum(O * dout) w.r.t. the un-rotated q, k, v.

    Per head: P from the forward definition, dv_j += sum_i P_ij dO_i,
    dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - sum_l P_il dP_il) (softmax
    Jacobian), d(Rq)_i = scale sum_j dS_ij (R k)_j,
    d(Rk)_j += scale sum_i dS_ij (R q)_i; finally dq = R^T d(Rq),
    dk = R^T d(Rk). Query heads of one kv group add into that group's dk/dv.
    With ``rows`` given, only those query rows contribute (dq is zero
    elsewhere and dk/dv hold those rows' contributions only).
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    rows = np.arange(prob.T) if rows is None else np.asarray(rows, dtype=np.int64)
    qr, kr = prob.rotated(q, k)
    allowed = mask_rows(rows, prob.doc, prob.mask_mode)
    dqr = np.zeros_like(q)
    dkr = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(prob.Hq):
        g = prob.kv_head(h)
        s = prob.scale * (qr[rows, h, :] @ kr[:, g, :].T)
        s = np.where(allowed, s, -np.inf)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)
        do = dout[rows, h, :]
        dv[:, g, :] += P.T @ do
        dP = do @ v[:, g, :].T
        dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
        dqr[rows, h, :] = prob.scale * (dS @ kr[:, g, :])
        dkr[:, g, :] += prob.scale * (dS.T @ qr[rows, h, :])
    dq = rotate(dqr, prob.pos, prob.base, prob.layout, inverse=True, theta=prob.theta)
    dk = rotate(dkr, prob.pos, prob.base, prob.layout, inverse=True, theta=prob.theta)
    return dq, dk, dv
