"""CPU oracle for the video-DiT attention hot path (float64, numpy).

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this module. The CUDA
library never calls it, and it shares no code with the CUDA path: it imports
nothing from the package and the package imports nothing from here.

What it computes, and where the pages say so:

* Full, non-causal spatio-temporal self-attention over every latent token
  ("Wan Team, Alibaba (2025)" anthology note, *Key takeaways*: full
  spatio-temporal self-attention over latent patches; ctol.digital article,
  *Engineering the Core*).
* 3D RoPE on Q and K, with separate temporal / height / width bands (gojay.top
  "Wan2.1" reading, *费曼一分钟* and *DiT 块*: 3D RoPE gives the space-time
  positions).
* Tokens come from a (1,2,2) patchify of the latent: L = F * Hp * Wp
  (gojay.top reading, *DiT backbone*).
* Cross-attention from video tokens to at most 512 umT5 text tokens
  (gojay.top reading, *⑥ 1.3B vs 14B* config table and *符号速查表*;
  aipaper.jasonlin.tech summary, *Key contributions*: the 512-token limit).
* The backward pass that rectified-flow training needs (gojay.top reading,
  *§3 Training*).

The pages print no attention formula, no RoPE constants, no layout and no
worked example. Where they are silent this module takes the following
readings (each is also listed in the design notes):

R1  RoPE pairs are adjacent dims (2j, 2j+1) inside each band; the bands are
    contiguous in the order t, h, w with widths d - 4*(d//6), 2*(d//6),
    2*(d//6) (44/42/42 at d = 128).
R2  Band-local frequencies: pair j of a band of width d_b turns by
    pos * theta**(-2j/d_b); theta = 10000.
R3  Positions are the 0-based integer grid coordinates (t, h, w) of a token.
R4  Token order is row-major over (F, Hp, Wp): l = (t*Hp + h)*Wp + w.
R5  Logits are scale * <q_rot, k_rot> with scale = 1/sqrt(d); LSE is the
    natural log of sum_j exp(logit_ij) over valid keys.
R6  Cross-attention masks keys j >= kv_len[b]; a row with no valid key gives
    O = 0 and LSE = -inf.
R7  Everything is float64 here; no intermediate is rounded to bf16.

Parity pins (tests/test_oracle.py): brute-force loops on an 8-token grid,
Q = 0 -> mean(V), one-hot dominant logit, RoPE relative-offset invariance and
agreement with complex multiplication, positions-at-zero == textbook softmax
attention (scipy), central finite differences of the backward, gradient sum
invariants, and the two-part log-sum-exp merge identity.
"""
from __future__ import annotations

import math

import numpy as np

DEFAULT_THETA = 10000.0


# ---------------------------------------------------------------------------
# Token grid and 3D RoPE


def rope_bands(head_dim: int):
    """(offset, width) of the t, h and w bands of a head (reading R1)."""
    if head_dim % 2 or head_dim < 6:
        raise ValueError("head_dim must be even and >= 6")
    w_hw = 2 * (head_dim // 6)
    w_t = head_dim - 2 * w_hw
    return ((0, w_t), (w_t, w_hw), (w_t + w_hw, w_hw))


def token_coords(F: int, Hp: int, Wp: int):
    """(t, h, w) integer coordinates of every token, in token order (R3, R4)."""
    l = np.arange(F * Hp * Wp, dtype=np.int64)
    w = l % Wp
    h = (l // Wp) % Hp
    t = l // (Wp * Hp)
    return t, h, w


def rope_angles(F: int, Hp: int, Wp: int, head_dim: int, theta: float = DEFAULT_THETA):
    """Rotation angle of every (token, rotary pair): float64 [L, head_dim/2] (R1-R3)."""
    coords = token_coords(F, Hp, Wp)
    L = F * Hp * Wp
    ang = np.zeros((L, head_dim // 2), dtype=np.float64)
    for (off, width), pos in zip(rope_bands(head_dim), coords):
        j = np.arange(width // 2, dtype=np.float64)
        omega = theta ** (-2.0 * j / width)
        ang[:, off // 2: off // 2 + width // 2] = pos[:, None].astype(np.float64) * omega[None, :]
    return ang


def rope_rotate(x: np.ndarray, angles: np.ndarray, inverse: bool = False) -> np.ndarray:
    """Turn each pair (x[2p], x[2p+1]) of every token by its angle.

    x: [..., L, d] float64, angles: [L, d/2]. The forward map is
    (a, b) -> (a cos - b sin, a sin + b cos); ``inverse`` applies the
    transpose (the angle negated), which is what the backward pass needs.
    """
    c = np.cos(angles)
    s = np.sin(angles)
    if inverse:
        s = -s
    a = x[..., 0::2]
    b = x[..., 1::2]
    out = np.empty_like(x, dtype=np.float64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


# ---------------------------------------------------------------------------
# Forward: explicit softmax matrix, one block of query rows at a time


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                      n_valid: int | None = None):
    """Plain attention for the query rows q [m, d] against keys k, v [n, d].

    Keys j >= n_valid are excluded (R6). Returns O [m, d] and LSE [m] (R5).
    The whole softmax row is formed explicitly for every query.
    """
    n = k.shape[0] if n_valid is None else min(int(n_valid), k.shape[0])
    m = q.shape[0]
    if n <= 0:
        return np.zeros((m, v.shape[1])), np.full(m, -np.inf)
    s = scale * (q @ k[:n].T)                       # logits [m, n]
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom                                   # softmax matrix rows
    o = p @ v[:n]
    lse = mx[:, 0] + np.log(denom[:, 0])
    return o, lse


def _row_blocks(n: int, block: int):
    for i0 in range(0, n, block):
        yield i0, min(n, i0 + block)


def self_attention_fwd(q, k, v, grid, theta=DEFAULT_THETA, scale=None, block=1024):
    """3D-RoPE self-attention over every query row.

    q, k, v: float64 [B, L, H, d] (token-major). grid = (F, Hp, Wp).
    Returns O [B, L, H, d] and LSE [B, H, L].
    """
    B, L, H, d = q.shape
    F, Hp, Wp = grid
    assert F * Hp * Wp == L
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    o = np.zeros((B, L, H, d))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            qr = rope_rotate(q[b, :, h, :], ang)
            kr = rope_rotate(k[b, :, h, :], ang)
            for i0, i1 in _row_blocks(L, block):
                o[b, i0:i1, h, :], lse[b, h, i0:i1] = softmax_attention(
                    qr[i0:i1], kr, v[b, :, h, :], scale)
    return o, lse


def self_attention_fwd_rows(q_rows, rows_bhi, k_head, v_head, grid, theta=DEFAULT_THETA,
                            scale=None):
    """Self-attention for selected query rows of ONE (b, h).

    q_rows: float64 [m, d] (pre-RoPE queries); rows_bhi: their token indices
    [m]; k_head, v_head: float64 [L, d] of that (b, h). Returns O [m, d], LSE [m].
    """
    L, d = k_head.shape
    F, Hp, Wp = grid
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    qr = rope_rotate(q_rows, ang[np.asarray(rows_bhi)])
    kr = rope_rotate(k_head, ang)
    return softmax_attention(qr, kr, v_head, scale)


def cross_attention_fwd(q, k, v, kv_lens, scale=None, block=4096):
    """Cross-attention (no RoPE) from video tokens to padded text keys.

    q: [B, Lq, H, d]; k, v: [B, Lk, H, d]; kv_lens: [B] valid key counts (R6).
    Returns O [B, Lq, H, d] and LSE [B, H, Lq].
    """
    B, Lq, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = np.zeros((B, Lq, H, d))
    lse = np.zeros((B, H, Lq))
    for b in range(B):
        for h in range(H):
            for i0, i1 in _row_blocks(Lq, block):
                o[b, i0:i1, h, :], lse[b, h, i0:i1] = softmax_attention(
                    q[b, i0:i1, h, :], k[b, :, h, :], v[b, :, h, :], scale, kv_lens[b])
    return o, lse


def decoupled_cross_attention_fwd(q, k_txt, v_txt, lens_txt, k_img, v_img, lens_img, scale=None):
    """Image-to-video cross-attention: the text path and the image path are
    attended separately and their outputs added ("Wan Team, Alibaba (2025)"
    anthology note, Key takeaways: a CLIP image embedding enters through
    decoupled cross-attention; gojay.top reading, code map (4) WanModel T2V /
    I2V: two attention paths, then summed). Returns O [B, Lq, H, d] and the
    text path's LSE [B, H, Lq].
    """
    o_t, lse_t = cross_attention_fwd(q, k_txt, v_txt, lens_txt, scale)
    o_i, _ = cross_attention_fwd(q, k_img, v_img, lens_img, scale)
    return o_t + o_i, lse_t


def self_attention_fwd_chunk(q_rows, q_start, k_chunk, v_chunk, kv_start, grid, theta=DEFAULT_THETA, scale=None):
    """Attention of consecutive query tokens over consecutive key tokens of one
    (b, h), with 3D RoPE at the tokens' own grid positions: the partial result
    one Ring-attention step produces (anthology note, Key takeaways: Ring
    Attention across devices in the 2D context parallelism).

    q_rows: [m, d] tokens q_start .. q_start+m-1; k_chunk, v_chunk: [n, d]
    tokens kv_start .. kv_start+n-1. Returns O [m, d] and LSE [m] over those
    n keys only.
    """
    m, d = q_rows.shape
    n = k_chunk.shape[0]
    F, Hp, Wp = grid
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    qr = rope_rotate(q_rows, ang[q_start:q_start + m])
    kr = rope_rotate(k_chunk, ang[kv_start:kv_start + n])
    return softmax_attention(qr, kr, v_chunk, scale)


# ---------------------------------------------------------------------------
# Backward (for the rectified-flow training step)


def _head_backward(qr_rows, do_rows, kr, vh, scale, block, need_dkdv=True):
    """Gradients of one head with rotated operands.

    qr_rows, do_rows: rotated queries and upstream gradients of the query rows
    to process [m, d]; kr, vh: rotated keys and values of the head [n, d].
    For every query row i:
      P_i = softmax(scale * qr_i . kr^T),  O_i = P_i v,  D_i = dO_i . O_i,
      dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
      dQr_i = scale * sum_j dS_ij kr_j,  dKr_j += scale * dS_ij qr_i,
      dV_j += P_ij dO_i.
    Returns dQ_rot [m, d] and, if asked, dK_rot and dV [n, d] summed over the
    processed rows.
    """
    m = qr_rows.shape[0]
    dqr = np.zeros((m, qr_rows.shape[1]))
    dkr = np.zeros_like(kr) if need_dkdv else None
    dv = np.zeros_like(vh) if need_dkdv else None
    for r0, r1 in _row_blocks(m, block):
        qb, dob = qr_rows[r0:r1], do_rows[r0:r1]
        s = scale * (qb @ kr.T)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        p = e / e.sum(axis=1, keepdims=True)
        o = p @ vh
        d_i = np.sum(dob * o, axis=1, keepdims=True)
        dp = dob @ vh.T
        ds = p * (dp - d_i)
        dqr[r0:r1] = scale * (ds @ kr)
        if need_dkdv:
            dkr += scale * (ds.T @ qb)
            dv += p.T @ dob
    return dqr, dkr, dv


def head_backward_given_o_lse(qr_rows, do_rows, kr, vh, o_rows, lse_rows, scale):
    """Gradients of one head as the backward entry point defines them: from the
    forward's outputs rather than recomputed ones.

    The backward is handed O and LSE by the forward; the softmax weights are
    P_ij = exp(scale * qr_i . kr_j - LSE_i) and the row term is
    D_i = dO_i . O_i with that O (gojay.top reading, section 3 Training: the
    gradient of the softmax through dS = P o (dP - D)). With the exact O and
    LSE this is _head_backward; with rounded ones it is the backward of the
    values a training step actually passes on.
    Returns dQ_rot [m, d], dK_rot [n, d], dV [n, d].
    """
    s = scale * (qr_rows @ kr.T)
    p = np.exp(s - lse_rows[:, None])
    d_i = np.sum(do_rows * o_rows, axis=1, keepdims=True)
    ds = p * (do_rows @ vh.T - d_i)
    return scale * (ds @ kr), scale * (ds.T @ qr_rows), p.T @ do_rows


def self_attention_bwd(q, k, v, dout, grid, theta=DEFAULT_THETA, scale=None, block=1024):
    """dQ, dK, dV [B, L, H, d] of sum(O * dout) for 3D-RoPE self-attention.

    The RoPE backward applies the transposed rotation to dQ_rot and dK_rot.
    """
    B, L, H, d = q.shape
    F, Hp, Wp = grid
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            qr = rope_rotate(q[b, :, h, :], ang)
            kr = rope_rotate(k[b, :, h, :], ang)
            dqr, dkr, dvh = _head_backward(qr, dout[b, :, h, :], kr, v[b, :, h, :], scale, block)
            dq[b, :, h, :] = rope_rotate(dqr, ang, inverse=True)
            dk[b, :, h, :] = rope_rotate(dkr, ang, inverse=True)
            dv[b, :, h, :] = dvh
    return dq, dk, dv


def self_attention_bwd_dq_rows(q_rows, do_rows, rows, k_head, v_head, grid,
                               theta=DEFAULT_THETA, scale=None, block=1024):
    """dQ of selected query rows of ONE (b, h).

    q_rows, do_rows: pre-RoPE queries and upstream gradients of those rows
    [m, d]; rows: their token indices; k_head, v_head: [L, d] of the head.
    """
    L, d = k_head.shape
    F, Hp, Wp = grid
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    rows = np.asarray(rows)
    qr = rope_rotate(q_rows, ang[rows])
    kr = rope_rotate(k_head, ang)
    dqr, _, _ = _head_backward(qr, do_rows, kr, v_head, scale, block, need_dkdv=False)
    return rope_rotate(dqr, ang[rows], inverse=True)


def self_attention_bwd_dkdv_rows(q_head, k_head, v_head, do_head, key_rows, grid, theta=DEFAULT_THETA,
                                 scale=None, block=64, row_map=map):
    """dK and dV of selected key rows of ONE (b, h).

    q_head, k_head, v_head, do_head: float64 [L, d] of the head (pre-RoPE);
    key_rows: the token indices J of the key rows wanted. Every query row
    contributes to a key row's gradient, so all L query rows are visited:
      1. the forward over all keys gives LSE_i and O_i of every query row,
         and D_i = dO_i . O_i;
      2. for the selected keys only, with P_ij = exp(scale qr_i . kr_j - LSE_i)
         (the softmax entries of column j), dP_ij = dO_i . v_j and
         dS_ij = P_ij (dP_ij - D_i):
           dKr_j = scale sum_i dS_ij qr_i,   dV_j = sum_i P_ij dO_i,
           dK_j = R(pos_j)^T dKr_j.
    These are the columns J of the full backward (self_attention_bwd).
    `row_map` maps the forward over blocks of query rows; the builtin map by
    default (a thread pool's map gives the same result, faster).
    Returns dK [|J|, d] and dV [|J|, d].
    """
    L, d = k_head.shape
    F, Hp, Wp = grid
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    ang = rope_angles(F, Hp, Wp, d, theta)
    key_rows = np.asarray(key_rows)
    qr = rope_rotate(q_head, ang)
    kr = rope_rotate(k_head, ang)

    def forward_block(bounds):
        i0, i1 = bounds
        return softmax_attention(qr[i0:i1], kr, v_head, scale)

    parts = list(row_map(forward_block, list(_row_blocks(L, block))))
    o = np.concatenate([p[0] for p in parts])
    lse = np.concatenate([p[1] for p in parts])
    d_i = np.sum(do_head * o, axis=1)
    kr_j, v_j = kr[key_rows], v_head[key_rows]
    dkr = np.zeros((len(key_rows), d))
    dv = np.zeros((len(key_rows), d))
    for i0, i1 in _row_blocks(L, 4096):
        p = np.exp(scale * (qr[i0:i1] @ kr_j.T) - lse[i0:i1, None])
        dp = do_head[i0:i1] @ v_j.T
        ds = p * (dp - d_i[i0:i1, None])
        dkr += scale * (ds.T @ qr[i0:i1])
        dv += p.T @ do_head[i0:i1]
    return rope_rotate(dkr, ang[key_rows], inverse=True), dv


# ---------------------------------------------------------------------------
# Partial results over disjoint key sets (the state a ring step carries)


def merge_partials(o_a, lse_a, o_b, lse_b):
    """Combine attention over key sets A and B into attention over A u B.

    With LSE the natural log-sum-exp of the scaled logits (R5), the weights of
    the two parts are exp(LSE_A) and exp(LSE_B):
      O = (e^LSE_A O_A + e^LSE_B O_B) / (e^LSE_A + e^LSE_B),
      LSE = log(e^LSE_A + e^LSE_B).
    """
    lse = np.logaddexp(lse_a, lse_b)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - np.where(np.isneginf(lse), 0.0, lse)))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - np.where(np.isneginf(lse), 0.0, lse)))
    return wa[..., None] * o_a + wb[..., None] * o_b, lse


def attention_flops(B, H, Lq, Lk, d, backward=False):
    """FLOP convention of the workload: 4*B*H*Lq*Lk*d forward, 2.5x for backward."""
    f = 4.0 * B * H * Lq * Lk * d
    return 2.5 * f if backward else f
