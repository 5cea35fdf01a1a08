"""Float64 CPU oracle for the Kimi Delta Attention (KDA) recurrent decode update.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, tables or helpers) and imports nothing from the
package.

Everything here is plain numpy in float64.  Inputs are the values as stored
(bfloat16 inputs are upcast exactly by the caller); no intermediate rounding
happens; results are returned in float64 and the tests compare the GPU's
rounded results against them.

Sources (web pages, cited by title and section):

* "flashinfer.kda_decode" (module overview page): the Kimi-Linear T=1 gate
  ``-exp(A_log) * softplus(g + dt_bias)`` with in-kernel beta sigmoid and QK
  normalisation (Cake T=1..6 family bullets); the split of packed QKV and the
  fixed ``lower_bound=-5`` transform (section "Serving-native packed Kimi K3
  decode"); null padding rows emit zero without touching state (same
  section); packed ``cu_seqlens`` with ragged lengths and null slots
  (section "Frozen / speculative-verify mode").
* "flashinfer.kda_decode.fused_kda_decode" (API page, "Parameters"): shapes of
  x, weight, conv_state, raw_gate, raw_beta, A_log, dt_bias, state_indices,
  state, output_gate, norm_weight; slot 0 is the null slot; non-positive rows
  produce zeros and update neither cache; the recurrence is evaluated in
  float32 and a bfloat16 state is rounded when written back.
* "feat(cake_kda): add serving-native packed decode backend" (section "Exact
  contract"): H=12, K=V=128, packed QKV [B, 4608], raw gate [B, 1536], raw
  beta [B, 12], scale 1/sqrt(128), L2 epsilon 1e-6, lower_bound -5, and -1
  as an inactive padding row.
* "feat(kda): add fused speculative decode kernel - #4809" (review thread on
  the T=1 row mapping): token rows past the last ``query_start_loc`` entry are
  padding that write zero and touch no slot; the packed fused operation
  updates conv and recurrent checkpoints from accepted-token metadata; its
  bf16-state follow-up keeps the recurrence in float32 across the token loop
  and rounds each per-token checkpoint on store.

Readings where the pages are silent (each is a named constant or flag below):

* State orientation: ``S[k][v]`` (row = key channel, column = value channel).
* Bounded gate: ``g = lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias))``.
  The pages name a "lower_bound gate transform" but print no formula, so the
  CHOICE of this formula is parity unpinned by the pages; the function itself
  is pinned to the identities that formula implies.
* L2 normalisation ``x * (sum(x^2) + eps)^-1/2`` with eps = 1e-6.
* Update order: decay, read ``S_d^T k``, delta write, output from the updated
  state.
* Conv taps: the three cached samples are oldest to newest and take weight
  taps 0..2, the new sample takes tap 3; the cache holds raw (pre-conv)
  samples; no bias; SiLU after the conv; weight sections in q, k, v order.
* Output gate: RMSNorm over the 128 channels of a head (eps inside the square
  root), times ``norm_weight``, times ``sigmoid(output_gate)``.
* Slot indices outside ``[1, num_slots)`` take the null path.
* Packed fused checkpoints: ``state_indices`` is [N, C]; sequence n starts
  from slot ``state_indices[n, num_accepted_tokens[n] - 1]`` and writes both
  caches after its j-th token to slot ``state_indices[n, j]`` (j < C); a
  non-live checkpoint slot is skipped; ``num_accepted_tokens`` outside 1..C
  makes the sequence null.
"""

from __future__ import annotations

import numpy as np

# --- constants fixed by the pages ---------------------------------------------------

D = 128                      # head dimension K = V = 128 ("Exact contract")
SCALE = 1.0 / np.sqrt(128.0)  # fixed output scale ("Exact contract")
L2_EPS = 1e-6                # QK L2 normalisation epsilon ("Exact contract")
PACKED_HEADS = 12            # Kimi K3 packed contract heads ("Exact contract")
PACKED_LOWER_BOUND = -5.0    # fixed lower_bound of the packed contract
FUSED_NORM_EPS = 1e-5        # default norm_eps of fused_kda_decode ("Parameters")
CONV_WIDTH = 4               # width-four depthwise causal convolution ("fused_kda_decode")

GATE_SOFTPLUS = "softplus"
GATE_LOWER_BOUND = "lower_bound"


# --- elementwise pieces --------------------------------------------------------------

def softplus(x):
    """log(1 + e^x), evaluated without overflow as max(x, 0) + log1p(e^-|x|)."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    """1 / (1 + e^-x), evaluated without overflow on either side."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def silu(x):
    """x * sigmoid(x): the activation after the short convolution."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def l2_normalize(x, eps=L2_EPS):
    """x * (sum(x^2) + eps)^(-1/2) over the last axis (QK normalisation, eps 1e-6)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gate_softplus(raw_g, dt_bias, A_log):
    """Kimi-Linear gate g = -exp(A_log[h]) * softplus(raw_g + dt_bias).

    "flashinfer.kda_decode", Cake T=1..6 family bullets (Kimi-Linear T=1
    equal-head schedules).  raw_g and dt_bias are [..., H, 128]; A_log is [H].
    """
    a = np.exp(np.asarray(A_log, dtype=np.float64))[..., :, None]
    return -a * softplus(np.asarray(raw_g, np.float64) + np.asarray(dt_bias, np.float64))


def gate_lower_bound(raw_g, dt_bias, A_log, lower_bound):
    """Bounded gate g = lower_bound * sigmoid(exp(A_log[h]) * (raw_g + dt_bias)).

    The pages name a "fixed lower_bound=-5 gate transform" ("Serving-native
    packed Kimi K3 decode") and a "negative lower bound used by the recurrence
    gate", distinct from the softplus gate ("fused_kda_decode", Parameters),
    but print no formula.  This reading keeps g in (lower_bound, 0).
    """
    a = np.exp(np.asarray(A_log, dtype=np.float64))[..., :, None]
    x = np.asarray(raw_g, np.float64) + np.asarray(dt_bias, np.float64)
    return float(lower_bound) * sigmoid(a * x)


def gate(raw_g, dt_bias, A_log, lower_bound):
    """Gate of the T=1 paths: softplus form when lower_bound is None, else bounded."""
    if lower_bound is None:
        return gate_softplus(raw_g, dt_bias, A_log)
    return gate_lower_bound(raw_g, dt_bias, A_log, lower_bound)


# --- the recurrent step --------------------------------------------------------------

def kda_step_u(S, q, k, v, g, beta, scale=SCALE):
    """One KDA decode step for one (row, head) unit, with its correction.

    S is the [K=128][V=128] state (row = key channel); q, k, v, g are [128]
    vectors with g the per-key-channel log decay; beta is the delta-rule
    learning rate.  Steps, in order: L2-normalise q and k; decay the state by
    diag(exp(g)); delta write S' = S_d + k u^T with the correction
    u = beta (v - S_d^T k); output o = scale * S'^T q.  Returns (S', o, u).
    """
    S = np.asarray(S, dtype=np.float64)
    qh = l2_normalize(q)
    kh = l2_normalize(k)
    Sd = np.exp(np.asarray(g, np.float64))[:, None] * S
    u = float(beta) * (np.asarray(v, np.float64) - Sd.T @ kh)
    S_new = Sd + np.outer(kh, u)
    o = scale * (S_new.T @ qh)
    return S_new, o, u


def kda_step(S, q, k, v, g, beta, scale=SCALE):
    """One KDA decode step (see kda_step_u); returns (S', o)."""
    S_new, o, _ = kda_step_u(S, q, k, v, g, beta, scale)
    return S_new, o


def _is_live(slot, num_slots):
    """Live slots are [1, num_slots); anything else takes the null path."""
    return 0 < int(slot) < int(num_slots)


# --- entry points --------------------------------------------------------------------

def recurrent_decode(q, k, v, raw_gate, raw_beta, A_log, dt_bias, state_indices,
                     state, lower_bound=None, scale=SCALE):
    """T=1 recurrent decode over B rows (one token per row).

    q, k, v, raw_gate: [B, H, 128]; raw_beta: [B, H]; A_log: [H];
    dt_bias: [H * 128]; state_indices: [B] ints; state: [N, H, 128, 128].
    Returns (out [B, H, 128], new_state [N, H, 128, 128]) in float64; rows
    whose slot is outside [1, N) give zero output and leave the pool alone.
    """
    q = np.asarray(q, np.float64)
    B, H, _ = q.shape
    state = np.array(state, dtype=np.float64, copy=True)
    N = state.shape[0]
    dt = np.asarray(dt_bias, np.float64).reshape(H, D)
    out = np.zeros((B, H, D), dtype=np.float64)
    for b in range(B):
        s = int(state_indices[b])
        if not _is_live(s, N):
            continue
        g = gate(np.asarray(raw_gate[b], np.float64), dt, A_log, lower_bound)
        beta = sigmoid(np.asarray(raw_beta[b], np.float64))
        for h in range(H):
            state[s, h], out[b, h] = kda_step(state[s, h], q[b, h], k[b, h], v[b, h],
                                              g[h], beta[h], scale)
    return out, state


def split_packed_qkv(mixed_qkv, heads=PACKED_HEADS):
    """Split post-conv packed QKV [B, 3*H*128] into q, k, v of [B, H, 128] each.

    "Exact contract": packed QKV [B, 4608] = three head-major 1536-wide blocks.
    """
    m = np.asarray(mixed_qkv, np.float64)
    B = m.shape[0]
    w = heads * D
    return (m[:, 0:w].reshape(B, heads, D), m[:, w:2 * w].reshape(B, heads, D),
            m[:, 2 * w:3 * w].reshape(B, heads, D))


def packed_decode(mixed_qkv, raw_gate, raw_beta, A_log, dt_bias, state_indices, state):
    """Kimi K3 packed T=1 decode: H=12, lower_bound -5, scale 1/sqrt(128).

    raw_gate [B, 1536] and raw_beta [B, 12] are viewed as [B, 12, 128] and
    [B, 12].  Returns (out [B, 12, 128], new_state).
    """
    q, k, v = split_packed_qkv(mixed_qkv)
    B = q.shape[0]
    rg = np.asarray(raw_gate, np.float64).reshape(B, PACKED_HEADS, D)
    return recurrent_decode(q, k, v, rg, raw_beta, A_log, dt_bias, state_indices,
                            state, lower_bound=PACKED_LOWER_BOUND)


def conv_silu_step(window, weight_taps):
    """Depthwise width-4 causal conv over one window, then SiLU.

    window: [C, 4] samples oldest to newest (3 cached + the new one);
    weight_taps: [C, 4] taps in the same order.  Returns [C].
    """
    y = np.sum(np.asarray(window, np.float64) * np.asarray(weight_taps, np.float64), axis=1)
    return silu(y)


def conv_weight_taps(weight):
    """Weight [3, 4, H*128] (section, tap, channel) as [3*H*128, 4] per channel."""
    w = np.asarray(weight, np.float64)
    return np.concatenate([w[sec].T for sec in range(w.shape[0])], axis=0)


def conv_update(x_row, weight, cache_slot):
    """One decode step of the short conv for one row: returns (a, new_cache).

    x_row: [3*H*128] new samples; weight: [3, 4, H*128]; cache_slot:
    [3*H*128, 3] cached raw samples oldest to newest.  a = SiLU(conv) over
    the window [cache, x]; the new cache drops the oldest sample and appends
    the raw x ("fused_kda_decode", Parameters: x, weight, conv_state).
    """
    x_row = np.asarray(x_row, np.float64)
    window = np.concatenate([np.asarray(cache_slot, np.float64), x_row[:, None]], axis=1)
    a = conv_silu_step(window, conv_weight_taps(weight))
    return a, window[:, 1:]


def gated_rmsnorm(o, output_gate, norm_weight, eps=FUSED_NORM_EPS):
    """RMSNorm over the last axis (128 channels) times weight, gated by sigmoid(logit)."""
    o = np.asarray(o, np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * np.asarray(norm_weight, np.float64) * sigmoid(output_gate)


def fused_decode(x, weight, conv_state, raw_gate, raw_beta, A_log, dt_bias,
                 state_indices, state, output_gate, norm_weight,
                 lower_bound=PACKED_LOWER_BOUND, norm_eps=FUSED_NORM_EPS):
    """Conv + SiLU, one KDA step and gated RMSNorm ("fused_kda_decode").

    x: [rows, 3*H*128]; weight: [3, 4, H*128]; conv_state: logical
    [N, 3*H*128, 3] (index [slot, channel, tap]); raw_gate: [rows, H, 128];
    raw_beta: [rows, H]; output_gate: [rows, H, 128]; norm_weight: [128];
    state: [N, H, 128, 128].  Returns (out [rows, H, 128], new_state,
    new_conv_state).  Null rows give zeros and touch neither cache.
    """
    x = np.asarray(x, np.float64)
    rows, C = x.shape
    H = C // (3 * D)
    HD = H * D
    state = np.array(state, dtype=np.float64, copy=True)
    conv_state = np.array(conv_state, dtype=np.float64, copy=True)
    N = state.shape[0]
    dt = np.asarray(dt_bias, np.float64).reshape(H, D)
    out = np.zeros((rows, H, D), dtype=np.float64)
    for r in range(rows):
        s = int(state_indices[r])
        if not _is_live(s, N):
            continue
        a, conv_state[s] = conv_update(x[r], weight, conv_state[s])
        q = a[0:HD].reshape(H, D)
        k = a[HD:2 * HD].reshape(H, D)
        v = a[2 * HD:3 * HD].reshape(H, D)
        g = gate(np.asarray(raw_gate[r], np.float64), dt, A_log, lower_bound)
        beta = sigmoid(np.asarray(raw_beta[r], np.float64))
        o = np.zeros((H, D))
        for h in range(H):
            state[s, h], o[h] = kda_step(state[s, h], q[h], k[h], v[h], g[h], beta[h])
        out[r] = gated_rmsnorm(o, np.asarray(output_gate[r], np.float64), norm_weight, norm_eps)
    return out, state, conv_state


def spec_decode(q, k, v, g, beta, cu_seqlens, state_indices, state,
                beta_is_logit=True, scale=SCALE):
    """Packed speculative decode: T >= 1 tokens per row with ragged cu_seqlens.

    q, k, v, g: [R, H, 128] token rows (g is the precomputed log decay);
    beta: [R, H] (logits when beta_is_logit, else the rate itself);
    cu_seqlens: [N+1]; state_indices: [N]; state: [M, H, 128, 128].
    Row n owns token rows cu[n] .. cu[n+1]-1, processed in order with the
    state carried in float64; the final state goes back to the row's slot.
    Token rows of null rows, and rows outside [cu[0], cu[N]), are zero.
    Returns (out [R, H, 128], new_state).
    """
    q = np.asarray(q, np.float64)
    R, H, _ = q.shape
    state = np.array(state, dtype=np.float64, copy=True)
    M = state.shape[0]
    rate = np.asarray(beta, np.float64)
    if beta_is_logit:
        rate = sigmoid(rate)
    out = np.zeros((R, H, D), dtype=np.float64)
    n_rows = len(state_indices)
    for n in range(n_rows):
        s = int(state_indices[n])
        t0, t1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        if not _is_live(s, M) or t1 <= t0:
            continue
        for h in range(H):
            S = state[s, h]
            for t in range(t0, t1):
                S, out[t, h] = kda_step(S, q[t, h], k[t, h], v[t, h], g[t, h], rate[t, h], scale)
            state[s, h] = S
    return out, state


def start_slot(row_slots, accepted):
    """The slot a packed fused sequence starts from: the checkpoint of its
    last accepted token, column accepted - 1 of its slot row."""
    return int(row_slots[int(accepted) - 1])


def packed_fused_decode(x, weight, conv_state, raw_gate, raw_beta, A_log, dt_bias,
                        state_indices, query_start_loc, num_accepted_tokens, state,
                        output_gate, norm_weight, lower_bound=PACKED_LOWER_BOUND,
                        norm_eps=FUSED_NORM_EPS, scale=SCALE):
    """Packed fused speculative decode with per-token checkpoints.

    "feat(kda): add fused speculative decode kernel - #4809" (description and
    the review thread on the T=1 row mapping) and its bf16-state follow-up:
    the fused conv + KDA + gated-RMSNorm step of ``fused_decode`` run over the
    T >= 1 token rows of each packed sequence, updating the conv and
    recurrent caches from accepted-token metadata.

    x: [R, 3*H*128] token rows; raw_gate, output_gate: [R, H, 128];
    raw_beta: [R, H]; state_indices: [N, C] checkpoint slots per sequence;
    query_start_loc: [N+1]; num_accepted_tokens: [N]; conv_state [M, 3*H*128, 3]
    and state [M, H, 128, 128] are slot-indexed pools.

    Sequence n owns token rows query_start_loc[n] .. query_start_loc[n+1]-1.
    It starts from the caches of slot state_indices[n, a-1], a =
    num_accepted_tokens[n] (the checkpoint of the last token accepted by the
    previous step); after its j-th token (j < C) both caches are written to
    slot state_indices[n, j] unless that slot is not live.  A sequence whose
    start slot is not live, or whose a is outside 1..C, is null: zero output,
    no cache written.  Rows outside [query_start_loc[0], query_start_loc[N])
    are padding: zero output.  The state is carried in float64 across tokens
    (the kernel's float32 registers); checkpoints are the carried values.
    Returns (out [R, H, 128], new_state, new_conv_state).
    """
    x = np.asarray(x, np.float64)
    R, C3 = x.shape
    H = C3 // (3 * D)
    HD = H * D
    state = np.array(state, dtype=np.float64, copy=True)
    conv_state = np.array(conv_state, dtype=np.float64, copy=True)
    M = state.shape[0]
    idx = np.asarray(state_indices).reshape(len(num_accepted_tokens), -1)
    n_seq, cols = idx.shape
    dt = np.asarray(dt_bias, np.float64).reshape(H, D)
    out = np.zeros((R, H, D), dtype=np.float64)
    for n in range(n_seq):
        t0 = max(int(query_start_loc[n]), 0)
        t1 = min(int(query_start_loc[n + 1]), R)
        acc = int(num_accepted_tokens[n])
        if t1 <= t0 or not 1 <= acc <= cols:
            continue
        s0 = start_slot(idx[n], acc)
        if not _is_live(s0, M):
            continue
        S = state[s0].copy()
        hist = conv_state[s0].copy()
        for j, t in enumerate(range(t0, t1)):
            a, hist = conv_update(x[t], weight, hist)
            q = a[0:HD].reshape(H, D)
            k = a[HD:2 * HD].reshape(H, D)
            v = a[2 * HD:3 * HD].reshape(H, D)
            g = gate(np.asarray(raw_gate[t], np.float64), dt, A_log, lower_bound)
            beta = sigmoid(np.asarray(raw_beta[t], np.float64))
            o = np.zeros((H, D))
            for h in range(H):
                S[h], o[h] = kda_step(S[h], q[h], k[h], v[h], g[h], beta[h], scale)
            out[t] = gated_rmsnorm(o, np.asarray(output_gate[t], np.float64), norm_weight, norm_eps)
            if j < cols and _is_live(int(idx[n, j]), M):
                state[int(idx[n, j])] = S
                conv_state[int(idx[n, j])] = hist
    return out, state, conv_state


def spec_verify(q, k, v, g, beta, cu_seqlens, state_indices, state, t_cap,
                beta_is_logit=True, scale=SCALE):
    """Speculative-verify mode: the spec_decode outputs from a read-only state.

    "flashinfer.kda_decode", section "Frozen / speculative-verify mode": the
    committed state is never written; slot-indexed out-params record, for
    token position t < t_cap of each live row, the delta-rule correction u_t
    ([M, H, t_cap, 128]) and the token's raw key followed by its log decay
    ([M, H, t_cap, 256]), for a later commit of the accepted tokens.
    Returns (out [R, H, 128], correction, kg); untouched entries are zero.
    """
    q = np.asarray(q, np.float64)
    R, H, _ = q.shape
    state = np.asarray(state, dtype=np.float64)
    M = state.shape[0]
    rate = np.asarray(beta, np.float64)
    if beta_is_logit:
        rate = sigmoid(rate)
    out = np.zeros((R, H, D))
    corr = np.zeros((M, H, t_cap, D))
    kg = np.zeros((M, H, t_cap, 2 * D))
    for n in range(len(state_indices)):
        s = int(state_indices[n])
        t0, t1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        if not _is_live(s, M) or t1 <= t0:
            continue
        for h in range(H):
            S = state[s, h]
            for t in range(t0, t1):
                S, out[t, h], u = kda_step_u(S, q[t, h], k[t, h], v[t, h], g[t, h], rate[t, h], scale)
                if t - t0 < t_cap:
                    corr[s, h, t - t0] = u
                    kg[s, h, t - t0, :D] = k[t, h]
                    kg[s, h, t - t0, D:] = g[t, h]
    return out, corr, kg


def commit_from_cache(S, kg_rows, corr_rows):
    """State after replaying cached tokens: S <- diag(exp(g)) S + k_hat u^T per token.

    kg_rows: [a, 256] raw key | log decay; corr_rows: [a, 128] corrections.
    """
    S = np.array(S, dtype=np.float64, copy=True)
    for kg_t, u in zip(kg_rows, corr_rows):
        kh = l2_normalize(kg_t[:D])
        S = np.exp(kg_t[D:])[:, None] * S + np.outer(kh, u)
    return S


# --- rounding helpers used by the tests ----------------------------------------------

def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significand bits); min normal spacing at 0."""
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)
