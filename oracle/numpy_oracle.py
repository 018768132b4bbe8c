"""Independent float64 NumPy restatement of the MoE-FFN forward layer (test
infrastructure only).

The oracle proper is the C++ library in this folder; this module restates the
same steps a second way (library matmul, argsort, exp and erf as steps, no
blocking, fusion or reordering) and serves only as one more pin of it
(``tests/test_oracle_cross.py``).  No value the C++ oracle produces comes from
here.  Page keys [P1]..[P5] are defined in ``oracle/__init__.py``.

Inputs are the exact values the device receives (bf16 bit patterns or
float32), widened exactly to float64.  Probabilities are computed in float64
and rounded to float32 before any decision (top-k, reroute order), because the
device takes those decisions on float32 probabilities.

Readings taken where the pages are silent or disagree (each also listed in
the design notes):
  R1 top-k ties go to the lower expert index ([P1] §5.5 asks for a stable top-k).
  R2 capacity C = floor(floor(k*N/E) * alpha) ([P1] §3.1 formula, §5.3 example).
  R3 drop keeps the first C assignments of an expert in ascending token order,
     whatever their slot ([P1] §4.2 code); a dropped slot contributes zero and
     its weight is not redistributed.
  R4 reroute ("next-best unfilled expert"): rounds; in each round every pending
     slot proposes the best expert (by probability, ties to the lower index)
     that was not full at the start of the round and that its token does not
     already hold or propose this round, slots of a token taken in slot order;
     each expert accepts proposals in ascending (token, slot) order while it
     has room.  A slot with no such expert is dropped.  A rerouted slot keeps
     its renormalised gate weight.  Inside an expert, primary assignments come
     first (token order), then reroutes in (round, token, slot) order.
  R5 load-balance statistics use [P3] §2.2's form on pre-capacity top-k picks:
     freq_e = picks_e/(N*k), P_e = mean_t p[t,e], L_bal = E * sum_e freq_e*P_e.
  R6 SwiGLU expert: silu(x Wg^T) * (x Wu^T), then Wd; silu(a) = a/(1+e^-a).
  R7 GELU is the erf form, nn.GELU()'s default ([P5] §3 code).
  R13 router z-loss ([P2] §3.3): L_z = 0.001 * mean_t logsumexp_e(z[t,e])^2 on
     the router's own logits z = x W_r^T, without the per-expert bias (the
     bias is not part of the router's linear map).
  R14 router entropy ([P4] §2.3 and its §3.1 code): per token, the softmax of
     the k selected logits (= the renormalised gates w), H_t = -sum_j w_j
     log2 w_j in bits (the page's code uses log2; its 1e-8 guard is left out,
     0 log 0 = 0), averaged over the tokens.
  R15 selection-only bias ([P5] §2.4, DeepSeek-V3): the expert bias steers the
     choice but leaves the router's probabilities alone: p = softmax(z), the
     top-k is taken on the float32 key p + b (ties to the lower index), the
     gates renormalise the unbiased p, mean_prob uses p, and reroute ranks
     candidates by the key.  The per-batch update lowers b_e by gamma when
     expert e got more than N*k/E pre-capacity picks and raises it by gamma
     when it got fewer (float32 arithmetic); the pages give no gamma.
  R16 low-precision expert weights ([P1] §5.4, [P4] §4.4: per-expert scales,
     the router stays in high precision): FP8 E4M3 (OCP 8-bit floating point
     format: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals,
     no infinities, S.1111.111 is NaN, largest finite 448).  One float32 scale
     per expert matrix, scale = amax/448 (1 for an all-zero matrix); a code is
     round-to-nearest-even of the float32 quotient w/scale, saturated to
     +-448.  Weights only: activations, accumulation and the SwiGLU product
     stay as in the bf16 layer; the dequantised weight is scale * code value.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

__all__ = [
    "widen", "router_logits", "softmax_fp32", "topk_select", "topk_margin",
    "renormalise", "balance_stats", "alpha_for_batch", "capacity",
    "apply_capacity_drop", "apply_capacity_reroute", "route", "dispatch",
    "gelu_erf", "silu", "expert_ffn", "combine_token", "moe_forward",
    "router_z_loss", "router_entropy", "selection_keys", "router_bias_update",
    "e4m3_encode", "e4m3_decode", "quantize_fp8", "dequantize_fp8",
]

# Parity pins: which CPU test pins each function to something other than itself.
PINS = {
    "router_logits": "tests/test_oracle_router.py: E=k special case, zero router, "
                     "permutation of experts; matmul is a library primitive",
    "softmax_fp32": "tests/test_oracle_router.py: scipy.special.softmax, shift invariance",
    "topk_select": "tests/test_oracle_router.py: brute force over all C(E,k) subsets",
    "renormalise": "tests/test_oracle_router.py: sum to 1, E=k gives w=p, golden case",
    "balance_stats": "tests/test_oracle_stats.py: L_bal=1 under uniform routing "
                     "([P3] §2.2), golden hand case",
    "capacity": "tests/test_oracle_capacity.py: [P1] §5.3 worked example C=1, "
                "[P5] exercise 1 (250), workload values 1280 / 2048",
    "apply_capacity_drop": "tests/test_oracle_capacity.py: counts<=C, all-to-one keeps "
                           "lowest tokens, C>=N*k is identity, golden hand case",
    "apply_capacity_reroute": "tests/test_oracle_reroute.py: hand-worked golden case, "
                              "counts<=C, no duplicate expert, next-best and "
                              "maximality properties",
    "expert_ffn": "tests/test_oracle_ffn.py: erf/exp special values, E=1 dense FFN",
    "router_z_loss": "tests/test_oracle_next.py: zero logits give 0.001*(ln E)^2, "
                     "scipy.special.logsumexp, shift by c adds c to lse",
    "router_entropy": "tests/test_oracle_next.py: equal gates give log2 k, one gate "
                      "gives 0, hand case (0.75, 0.25) -> 0.8112781 bits",
    "selection_keys": "tests/test_oracle_next.py: zero bias reduces to the plain "
                      "router, brute force over subsets of p+b, gates from unbiased p",
    "router_bias_update": "tests/test_oracle_next.py: hand case of signs, balanced "
                          "picks leave the bias unchanged",
    "e4m3_encode": "tests/test_oracle_fp8.py: torch float8_e4m3fn cast (library) on "
                   "random, tie and subnormal values; saturation and signed zero by hand",
    "e4m3_decode": "tests/test_oracle_fp8.py: all 256 codes vs torch float8_e4m3fn, "
                   "encode(decode(c)) == c for every finite code",
    "quantize_fp8": "tests/test_oracle_fp8.py: largest element maps to 448, error "
                    "<= half a step, zero matrix, hand case",
    "dequantize_fp8": "tests/test_oracle_fp8.py: product of the decoded code and the scale",
    "moe_forward": "tests/test_oracle_forward.py: E=1 dense layer, shared-only dense "
                   "layer, k=E layer = probability-weighted dense mixture of every "
                   "expert (logit and selection-only bias; a gate rotated to the "
                   "wrong expert fails), token-permutation equivariance, linearity "
                   "in the routed outputs, dropped slots contribute nothing; no page "
                   "prints a numeric layer output, so the pins are these special "
                   "cases and invariants",
}


# ----------------------------------------------------------------------------- inputs

def widen(a):
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------- router

def router_logits(x, w_router, router_bias=None):
    """z[t,e] = sum_j x[t,j] * Wr[e,j] (+ b[e]).

    [P5] §2.2: the router is a bias-free linear map d_model -> n_experts
    (``router_linear(x)``, ``nn.Linear(d_model, n_experts, bias=False)``).
    [P3] §2.2 TopKRouter: a per-expert ``expert_bias`` is added to the logits
    before the softmax; it takes no gradient.
    """
    z = widen(x) @ widen(w_router).T
    if router_bias is not None:
        z = z + widen(router_bias)[None, :]
    return z


def softmax_fp32(z):
    """p = softmax(z) over experts, in float64, rounded to float32.

    [P5] §2.2 ``expert_probs = softmax(router_logits)``; [P2] §2.2 G(x) =
    Softmax(x W_g).  exp(z - max z) / sum is the same function (shift invariance).
    """
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def topk_select(p, k):
    """Indices of the k largest probabilities per token, largest first (slot 0).

    [P5] §2.2 ``torch.topk(expert_probs, k)``.  Ties go to the lower expert
    index (reading R1): a stable sort of -p keeps equal values in index order.
    """
    order = np.argsort(-np.asarray(p, dtype=np.float32), axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def topk_margin(p, k):
    """Smallest gap between consecutive float32 scores among the k+1 largest
    (among all E when k == E), per token.

    Used to flag near-ties: a token whose gap is below 1e-6 may legitimately
    select a different set, or order its selected experts differently, on
    hardware that rounds the scores differently."""
    p = np.asarray(p, dtype=np.float32).astype(np.float64)
    E = p.shape[1]
    s = -np.sort(-p, axis=1)[:, :min(k + 1, E)]
    if s.shape[1] < 2:
        return np.full(p.shape[0], np.inf)
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


def renormalise(p, idx):
    """w[t,j] = p[t,idx_j] / sum_j' p[t,idx_j'], float64 then float32.

    [P5] §2.2 ``top_k_probs / top_k_probs.sum(dim=-1, keepdim=True)``; the
    page's rationale: the kept mass may be far below 1.  [P3] §2.2 does the same.
    """
    sel = np.take_along_axis(np.asarray(p, dtype=np.float32), idx.astype(np.int64), axis=1)
    sel = sel.astype(np.float64)
    return (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)


def balance_stats(p, idx, n_experts):
    """(expert_freq[E], mean_prob[E], L_bal) -- [P3] §2.2 ``load_balance_loss``.

    freq_e = #{(t,j): idx[t,j]=e} / (N*k)   (one-hot of the top-k picks)
    P_e    = (1/N) sum_t p[t,e]             (mean routing probability)
    L_bal  = E * sum_e freq_e * P_e          (equals 1 under uniform routing)
    """
    N, k = idx.shape
    freq = np.bincount(idx.ravel().astype(np.int64), minlength=n_experts) / float(N * k)
    mean_prob = np.asarray(p, dtype=np.float32).astype(np.float64).mean(axis=0)
    return freq, mean_prob, float(n_experts * np.sum(freq * mean_prob))


def router_z_loss(z):
    """L_z = 0.001 * mean_t (logsumexp_e z[t,e])^2 -- [P2] §3.3 (reading R13).

    z are the router's logits without the expert bias.  logsumexp is written
    out as m + log(sum exp(z - m)) with m the row maximum (the same function).
    """
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    return 0.001 * float(np.mean(lse * lse)) if len(lse) else 0.0


def router_entropy(w):
    """Mean over tokens of H_t = -sum_j w_j log2 w_j, bits -- [P4] §2.3 (reading R14).

    w are the renormalised top-k gates (the softmax of the selected logits).
    """
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    if w.shape[0] == 0:
        return 0.0
    terms = np.where(w > 0, -w * np.log2(np.where(w > 0, w, 1.0)), 0.0)
    return float(np.mean(terms.sum(axis=1)))


def selection_keys(p, router_bias):
    """key[t,e] = p[t,e] + b[e] in float32 -- [P5] §2.4 (reading R15)."""
    return (np.asarray(p, dtype=np.float32) +
            np.asarray(router_bias, dtype=np.float32)[None, :]).astype(np.float32)


def router_bias_update(router_bias, picks, n_tokens, k, gamma):
    """b_e - gamma if picks_e > N*k/E, b_e + gamma if picks_e < N*k/E -- [P5] §2.4.

    picks are the pre-capacity top-k picks per expert; float32 arithmetic.
    """
    b = np.asarray(router_bias, dtype=np.float32).copy()
    picks = np.asarray(picks, dtype=np.int64)
    E = len(b)
    g = np.float32(gamma)
    for e in range(E):
        load = picks[e] * E            # compare picks_e with N*k/E without division
        if load > n_tokens * k:
            b[e] = np.float32(b[e] - g)
        elif load < n_tokens * k:
            b[e] = np.float32(b[e] + g)
    return b


def route(x, w_router, router_bias, k, bias_mode=0):
    """Router stage: logits, float32 probabilities, top-k, gates, statistics.

    bias_mode 0: the expert bias is added to the logits before the softmax
    ([P3] §2.2); 1: the bias only steers the selection (reading R15).  "key" is
    what the top-k and the reroute rank by.
    """
    z_raw = router_logits(x, w_router, None)
    if bias_mode == 1 and router_bias is not None:
        p = softmax_fp32(z_raw)
        key = selection_keys(p, router_bias)
    else:
        p = softmax_fp32(router_logits(x, w_router, router_bias))
        key = p
    idx = topk_select(key, k)
    w = renormalise(p, idx)
    freq, mean_prob, l_bal = balance_stats(p, idx, p.shape[1])
    picks = np.bincount(idx.ravel().astype(np.int64), minlength=p.shape[1])
    return {"logits": z_raw, "p": p, "key": key, "idx": idx, "w": w,
            "margin": topk_margin(key, k), "expert_freq": freq, "mean_prob": mean_prob,
            "l_bal": l_bal, "picks": picks, "z_loss": router_z_loss(z_raw),
            "router_entropy": router_entropy(w)}


# ----------------------------------------------------------------------------- fp8 weights

E4M3_MAX = 448.0


def e4m3_encode(v):
    """float32 values -> FP8 E4M3 codes (uint8), round to nearest even, saturated.

    Reading R16.  Normal numbers are (1 + m/8) * 2^(e-7) for exponent field
    e = 1..15 and mantissa m = 0..7 (e = 15, m = 7 is NaN); subnormals are
    m * 2^-9.  A magnitude at or above 448 saturates to 448.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9 (a result of 8 is the smallest normal, code 8)
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)
    nrm = ~sub & (a < E4M3_MAX)
    if np.any(nrm):
        _, ex = np.frexp(a[nrm])             # a = f * 2^ex, f in [0.5, 1)
        e = ex - 1                           # a in [2^e, 2^(e+1))
        m = np.rint(a[nrm] / 2.0 ** (e - 3)).astype(np.int64)   # 8 .. 16
        carry = m == 16
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 8, m)
        code[nrm] = ((e + 7) << 3) | (m - 8)
    code[a >= E4M3_MAX] = 0x7E
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(code):
    """FP8 E4M3 codes -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return s * mag


def quantize_fp8(w):
    """One expert matrix (bf16 bit patterns or float32) -> (codes uint8, scale float32).

    scale = amax/448 in float32 (1 when the matrix is all zero); code =
    e4m3_encode(float32(w) / scale) with a float32 division (reading R16).
    """
    wf = widen(w).astype(np.float32)
    amax = np.float32(np.max(np.abs(wf))) if wf.size else np.float32(0)
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    return e4m3_encode((wf / scale).astype(np.float32)), scale


def dequantize_fp8(codes, scale):
    """scale * value(code), float64 (exact)."""
    return e4m3_decode(codes) * float(np.float32(scale))


# ----------------------------------------------------------------------------- capacity

def alpha_for_batch(n_tokens):
    """alpha = 1.0 + 0.5*log2(N/256) -- [P1] §3.1 tip (batch-dependent capacity factor)."""
    return 1.0 + 0.5 * math.log2(n_tokens / 256.0)


def capacity(n_tokens, n_experts, k, alpha):
    """C = floor( floor(k*N/E) * alpha ) -- [P1] §3.1 (reading R2).

    [P1] §5.3 works N=32, E=64, k=2, alpha=1.2 to capacity 1."""
    return int(math.floor(((k * n_tokens) // n_experts) * float(alpha)))


def apply_capacity_drop(idx, n_experts, cap):
    """Keep the first ``cap`` tokens of each expert in token order; drop the rest.

    [P1] §4.2 code: ``token_indices = torch.where(mask.any(-1))[0]`` (ascending)
    then ``token_indices[:expert_capacity]``.  [P5] §3 practice note: tokens
    over capacity are dropped.  ``cap=None`` means no limit.
    Returns (final_idx with -1 for dropped slots, members: per-expert token arrays).
    """
    N, k = idx.shape
    final = idx.astype(np.int32).copy()
    members = []
    for e in range(n_experts):
        hit = idx == e
        tokens = np.nonzero(hit.any(axis=1))[0]
        if cap is not None and len(tokens) > cap:
            over = tokens[cap:]
            final[over, np.argmax(hit[over], axis=1)] = -1
            tokens = tokens[:cap]
        members.append(tokens.astype(np.int32))
    return final, members


def apply_capacity_reroute(idx, p, n_experts, cap):
    """Drop, then reroute overflow to the next-best unfilled expert (reading R4).

    [P1] §3.1: tokens beyond an expert's capacity are forced to the next-best
    expert.  Returns (final_idx, members, n_rerouted, n_dropped, rounds).
    """
    N, k = idx.shape
    E = n_experts
    final, members = apply_capacity_drop(idx, E, cap)
    members = [list(m) for m in members]
    fill = np.array([len(m) for m in members], dtype=np.int64)
    order = np.argsort(-np.asarray(p, dtype=np.float32), axis=1, kind="stable")
    pending = [(t, j) for t in range(N) for j in range(k) if final[t, j] < 0]
    n_rerouted = 0
    n_dropped = 0
    rounds = 0
    while pending:
        rounds += 1
        full = fill >= cap                      # snapshot at the start of the round
        proposals = []                          # ((t, j), e) in ascending (t, j)
        proposed_by = {}
        for (t, j) in pending:
            taken = {int(final[t, jj]) for jj in range(k) if final[t, jj] >= 0}
            taken |= proposed_by.get(t, set())
            choice = -1
            for e in order[t]:
                if not full[e] and int(e) not in taken:
                    choice = int(e)
                    break
            if choice < 0:
                n_dropped += 1                  # nothing left: the slot stays dropped
                continue
            proposed_by.setdefault(t, set()).add(choice)
            proposals.append(((t, j), choice))
        still = []
        for (t, j), e in proposals:             # each expert accepts in (t, j) order
            if fill[e] < cap:
                final[t, j] = e
                members[e].append(t)
                fill[e] += 1
                n_rerouted += 1
            else:
                still.append((t, j))
        pending = still
    return final, [np.array(m, dtype=np.int32) for m in members], n_rerouted, n_dropped, rounds


def dispatch(idx, p, n_experts, cap_mode, cap):
    """Capacity stage.  cap_mode: 0 none, 1 drop, 2 reroute.

    Returns final_idx [N,k] (-1 = dropped), members (per-expert token lists in
    row order), counts [E], n_dropped, n_rerouted."""
    if cap_mode == 0:
        final, members = apply_capacity_drop(idx, n_experts, None)
        nr, nd = 0, 0
    elif cap_mode == 1:
        final, members = apply_capacity_drop(idx, n_experts, cap)
        nr, nd = 0, int((final < 0).sum())
    elif cap_mode == 2:
        final, members, nr, nd, _ = apply_capacity_reroute(idx, p, n_experts, cap)
    else:
        raise ValueError(cap_mode)
    counts = np.array([len(m) for m in members], dtype=np.int32)
    return {"final": final, "members": members, "counts": counts,
            "n_dropped": nd, "n_rerouted": nr}


# ----------------------------------------------------------------------------- experts

def gelu_erf(a):
    """GELU(a) = a * Phi(a) = 0.5 a (1 + erf(a/sqrt 2)) -- reading R7."""
    return 0.5 * a * (1.0 + _erf(a / math.sqrt(2.0)))


def silu(a):
    """silu(a) = a * sigmoid(a) = a / (1 + e^-a) -- reading R6 ([P1] §3.2 SwiGLU)."""
    return a / (1.0 + np.exp(-a))


def expert_ffn(x_rows, wts, act):
    """One expert applied to rows of x (float64 in, float64 out).

    act 0 (GELU, [P5] §3 ``Linear(d,d_ff) -> GELU -> Linear(d_ff,d)`` with biases):
        y = GELU(x W1^T + b1) W2^T + b2, W1 = wts['w_gate'] [F,d], W2 = wts['w_down'] [d,F]
    act 1 (SwiGLU, [P1] §3.2 ``Linear(d,4d) -> SwiGLU -> Linear(4d,d)``, reading R6):
        y = (silu(x Wg^T) * (x Wu^T)) Wd^T
    [P3] §2.3: shared experts are plain FFNs of the same form, not routed.
    """
    x = np.asarray(x_rows, dtype=np.float64)
    if act == 0:
        a = x @ widen(wts["w_gate"]).T
        if wts.get("b1") is not None:
            a = a + widen(wts["b1"])
        y = gelu_erf(a) @ widen(wts["w_down"]).T
        if wts.get("b2") is not None:
            y = y + widen(wts["b2"])
        return y
    g = x @ widen(wts["w_gate"]).T
    u = x @ widen(wts["w_up"]).T
    return (silu(g) * u) @ widen(wts["w_down"]).T


def combine_token(shared_rows, routed_rows, gates):
    """y_t = sum_s shared_s(x_t) + sum_j g_j * expert_j(x_t).

    [P5] §2.1 y = sum_i g_i(x) Expert_i(x); [P3] §2.3 the layer output is the
    shared-expert output plus the gate-weighted routed output.  Dropped slots
    carry gate 0 (reading R3)."""
    y = 0.0
    for r in shared_rows:
        y = y + r
    for g, r in zip(gates, routed_rows):
        y = y + float(g) * r
    return y


# ----------------------------------------------------------------------------- layer

def moe_forward(cfg, inputs, tokens=None, get_expert=None):
    """Whole layer: route, capacity, experts, combine, statistics.

    cfg: object with n_tokens, d_model, n_experts, top_k, d_ff, n_shared, act,
         cap_mode, alpha (the synth ``Workload`` fields).
    inputs: dict from ``synth.make_inputs`` (expert arrays may be omitted when
         ``get_expert(e)`` supplies one expert's weights on demand).
    tokens: indices of the tokens whose output rows to compute (default: all).
         Routing and capacity always run over the whole batch, since capacity
         couples the tokens of a batch; each output row then depends only on
         its own token.
    Returns a dict with routing tensors, statistics and y [len(tokens), d] float64.
    """
    N, E, k, S = cfg.n_tokens, cfg.n_experts, cfg.top_k, cfg.n_shared
    r = route(inputs["x"], inputs["w_router"], inputs.get("router_bias"), k,
              getattr(cfg, "bias_mode", 0))
    cap = capacity(N, E, k, cfg.alpha) if cfg.cap_mode != 0 else None
    dsp = dispatch(r["idx"], r["key"], E, cfg.cap_mode, cap)
    out = dict(r)
    out.update(dsp)
    out["capacity"] = cap

    if get_expert is None:
        def get_expert(e):
            return {key: (inputs[key][e] if inputs.get(key) is not None else None)
                    for key in ("w_gate", "w_up", "w_down", "b1", "b2")}

    tokens = np.arange(N) if tokens is None else np.asarray(tokens, dtype=np.int64)
    x = widen(inputs["x"])[tokens]
    final = dsp["final"][tokens]
    gates = r["w"][tokens]
    routed = {}                                   # (row in tokens, slot) -> expert output
    for e in range(E):
        rows, slots = np.nonzero(final == e)
        if len(rows) == 0:
            continue
        ye = expert_ffn(x[rows], get_expert(e), cfg.act)
        for i, (t, j) in enumerate(zip(rows, slots)):
            routed[(int(t), int(j))] = ye[i]
    shared = [expert_ffn(x, get_expert(E + s), cfg.act) for s in range(S)]
    y = np.zeros((len(tokens), cfg.d_model), dtype=np.float64)
    for t in range(len(tokens)):
        kept = [j for j in range(k) if final[t, j] >= 0]
        y[t] = combine_token([sh[t] for sh in shared],
                             [routed[(t, j)] for j in kept],
                             [gates[t, j] for j in kept])
    out["tokens"] = tokens
    out["y"] = y
    return out
