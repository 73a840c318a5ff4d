"""Plain CPU oracle for the forward pass of one sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU legs of bench.py
(cpu_baseline and --impl reference) may import this module. The CUDA library never calls it,
and it imports nothing from the CUDA path.

Everything is float64 numpy. Inputs arrive as the exact bf16 / fp32 values the GPU reads,
widened without rounding (see `bf16_bits_to_f64`). The method reaches a result with a plain
definition, so each function below is that definition written out, step by step, in the
order the pages give it:

  route    : logits = x . W_g ; selection score ; top-k ; softmax over the selected k
             ("大模型MoE稀疏激活原理与工程实践", §3.1 路由器, Router code: linear layer without
             bias, torch.topk(sorted=True), softmax over the top-k scores, weighted sum).
  bias     : selection on logits + expert_bias, gates from the unbiased logits
             ("AI架构演进从稀疏MoE到条件记忆的工程实践", gating-network code and its
             aux-loss-free bias term).
  gumbel   : g = -log(-log u), score = (logits + g) / tau
             ("GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token", §3.1 门控网络).
  capacity : capacity = tokens * k / E * capacity_factor, overflow slots marked and dropped
             ("参数规模与稀疏激活的真相拆解", §3.2 专家容量, Level 1 hard limit).
  reroute  : optional Level 2 of the same section: a dropped slot moves to the best-scoring
             expert that still has room and that its token does not already use.
  groups   : optional group-limited selection: keep the best groups of experts, then top-k
             inside them ("大模型MoE稀疏激活原理与工程实践", routing outlook).
  expert   : SwiGLU FFN  y = (silu(x W_gate) * (x W_up)) W_down
             ("GPT-4 ... 2% ...", §3.3 专家内部结构; "大模型MoE稀疏激活原理与工程实践", §3.2 专家).
  shared   : always-on shared experts added to the routed output
             ("V4" rework page, §2.2 混合专家层的设计细节).

Readings taken where the pages are silent or garbled (each one is listed with its reason in the
design notes of this repository):
  * ties in top-k go to the lower expert index; the selected experts are ordered by
    descending score, then ascending index;
  * BIAS mode gates come from the unbiased logits of the selected experts;
  * GUMBEL gates are a softmax over the selected perturbed scores (renormalised), no epsilons
    inside the logs (u is kept inside [2^-24, 1 - 2^-24] by the input generator);
  * capacity = ceil(cf * T * k / E) in exact rational arithmetic on the fp32 value of cf;
    slots claim capacity in token order (t ascending, then j); a dropped slot has gate 0 and
    the surviving gates are not renormalised;
  * shared experts have the routed experts' d_ff and gate weight 1; no residual is added.

Parity pins for every function live in tests/test_oracle_*.py (brute force, closed forms,
hand-worked fixtures under tests/golden/, and a dense every-expert path for the layer).
"""
from __future__ import annotations

from fractions import Fraction
import math

import numpy as np

PLAIN = 0
BIAS_SELECT = 1
GUMBEL = 2

TIE_MARGIN = 1e-5  # tokens whose adjacent top-(k+1) score gap is below this are exempt


# ----------------------------------------------------------------------------------------
# input widening
# ----------------------------------------------------------------------------------------
def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (a bf16 is the top half of a fp32)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 -> bf16 (round to nearest even via float32), return uint16 bit patterns.

    Used only to report the oracle's output at the layer's output precision.
    """
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


# ----------------------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------------------
def router_logits(x: np.ndarray, W_g: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_j x[t, j] * W_g[j, e]   (a linear layer with no bias)."""
    return np.asarray(x, np.float64) @ np.asarray(W_g, np.float64)


def gumbel_noise(u: np.ndarray) -> np.ndarray:
    """g = -log(-log(u)) evaluated in float64 on the given uniform samples."""
    u64 = np.asarray(u, dtype=np.float64)
    return -np.log(-np.log(u64))


def selection_scores(logits, mode, expert_bias=None, gumbel_u=None, tau=1.0) -> np.ndarray:
    """The score that top-k ranks.

    PLAIN       : s = logits
    BIAS_SELECT : s = logits + expert_bias[e]
    GUMBEL      : s = (logits + g) / tau,  g = -log(-log u)
    """
    logits = np.asarray(logits, np.float64)
    if mode == PLAIN:
        return logits.copy()
    if mode == BIAS_SELECT:
        return logits + np.asarray(expert_bias, np.float64)[None, :]
    if mode == GUMBEL:
        return (logits + gumbel_noise(gumbel_u)) / float(tau)
    raise ValueError(f"unknown routing mode {mode}")


def expert_order(s: np.ndarray) -> np.ndarray:
    """Per token, all experts sorted by descending score, ties by ascending expert index."""
    s = np.asarray(s, np.float64)
    T, E = s.shape
    order = np.empty((T, E), dtype=np.int64)
    for t in range(T):
        # a stable sort on -s keeps equal scores in ascending index order
        order[t] = np.argsort(-s[t], kind="stable")
    return order


def topk(s: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores, ordered by score (descending) then index (ascending)."""
    return expert_order(s)[:, :k].astype(np.int32)


def tie_margin(s: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between adjacent scores among each token's top-(k+1) sorted scores.

    A token whose margin is below TIE_MARGIN can legitimately flip between two correct
    fp32 evaluations of its logits; such tokens are exempt from the exact index check.
    """
    s = np.asarray(s, np.float64)
    srt = -np.sort(-s, axis=1)
    m = min(k + 1, s.shape[1])
    if m < 2:
        return np.full(s.shape[0], np.inf)
    return np.min(srt[:, : m - 1] - srt[:, 1:m], axis=1)


def group_limit(s: np.ndarray, n_groups: int, topk_groups: int) -> np.ndarray:
    """Two-level (group-limited) routing ("大模型MoE稀疏激活原理与工程实践", routing outlook: first
    pick one of 8 groups, then 2 experts inside it). Reading where the page is silent: experts
    e = 0..E-1 form n_groups consecutive groups of E / n_groups; a group's score is the largest
    selection score of its experts; the topk_groups best groups (ties to the lower group index)
    stay and every other expert's score becomes -inf, so top-k then picks inside them."""
    s = np.asarray(s, np.float64)
    T, E = s.shape
    size = E // n_groups
    out = np.full_like(s, -np.inf)
    for t in range(T):
        gs = [max(s[t, g * size:(g + 1) * size]) for g in range(n_groups)]
        order = sorted(range(n_groups), key=lambda g: (-gs[g], g))
        for g in order[:topk_groups]:
            out[t, g * size:(g + 1) * size] = s[t, g * size:(g + 1) * size]
    return out


def group_margin(s: np.ndarray, n_groups: int, topk_groups: int) -> np.ndarray:
    """Gap between the topk_groups-th and the next group score (inf when every group is kept)."""
    s = np.asarray(s, np.float64)
    T, E = s.shape
    if topk_groups >= n_groups:
        return np.full(T, np.inf)
    gs = -np.sort(-s.reshape(T, n_groups, E // n_groups).max(axis=2), axis=1)
    return gs[:, topk_groups - 1] - gs[:, topk_groups]


def gates(logits, s, idx, mode) -> np.ndarray:
    """Softmax over the k selected values.

    PLAIN / BIAS_SELECT: the selected *unbiased* logits.  GUMBEL: the selected perturbed scores.
    """
    src = np.asarray(s if mode == GUMBEL else logits, np.float64)
    a = np.take_along_axis(src, np.asarray(idx, np.int64), axis=1)
    a = a - a.max(axis=1, keepdims=True)
    ea = np.exp(a)
    return ea / ea.sum(axis=1, keepdims=True)


def route(x, W_g, k, mode=PLAIN, expert_bias=None, gumbel_u=None, tau=1.0, n_groups=0,
          topk_groups=0):
    """Full router: returns dict(logits, scores, topk_idx [T,k] int32, topk_w [T,k] f64, margin).

    With n_groups > 0 the selection is group-limited (see group_limit); `scores` are then the
    masked scores and `margin` also covers the group decision."""
    logits = router_logits(x, W_g)
    s = selection_scores(logits, mode, expert_bias, gumbel_u, tau)
    margin = None
    if n_groups > 0:
        margin = group_margin(s, n_groups, topk_groups)
        s = group_limit(s, n_groups, topk_groups)
    idx = topk(s, k)
    w = gates(logits, s, idx, mode)
    m = tie_margin(s, k)
    if margin is not None:
        m = np.minimum(m, margin)
    return {"logits": logits, "scores": s, "topk_idx": idx, "topk_w": w, "margin": m}


# ----------------------------------------------------------------------------------------
# capacity and permutation
# ----------------------------------------------------------------------------------------
def capacity(T: int, k: int, E: int, capacity_factor: float = 0.0, capacity_override: int = 0):
    """Per-expert slot limit, or None for no limit.

    capacity = (tokens * k) / E * capacity_factor, rounded up; an explicit positive override
    wins; a factor <= 0 means no limit.  The factor is taken at its fp32 value, exactly.
    """
    if capacity_override > 0:
        return int(capacity_override)
    cf = float(np.float32(capacity_factor))
    if cf <= 0.0:
        return None
    return int(math.ceil(Fraction(cf) * T * k / E))


def permute(topk_idx: np.ndarray, E: int, C=None):
    """Counting-sort definition of dispatch.

    Walk the slots in token order (t ascending, then j); slot (t, j) is index t*k + j. Each
    expert accepts slots until it holds C of them; later ones are dropped.  Kept slots are laid
    out expert by expert (offsets = exclusive scan of the kept counts), in arrival order.

    Returns counts [E] (before the limit), offsets [E+1], perm_slot [T*k] (position -> slot,
    -1 past the last kept position), slot_pos [T*k] (slot -> position, -1 when dropped).
    """
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    kept = counts.copy() if C is None else np.minimum(counts, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + kept[e]
    fill = np.zeros(E, dtype=np.int64)
    perm_slot = np.full(T * k, -1, dtype=np.int64)
    slot_pos = np.full(T * k, -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            if C is None or fill[e] < C:
                p = offsets[e] + fill[e]
                fill[e] += 1
                perm_slot[p] = t * k + j
                slot_pos[t * k + j] = p
    return {"counts": counts.astype(np.int32), "offsets": offsets.astype(np.int32),
            "perm_slot": perm_slot.astype(np.int32), "slot_pos": slot_pos.astype(np.int32),
            "n_kept": int(offsets[E])}


def permute_by_sort(topk_idx: np.ndarray, E: int, C=None):
    """Second, independent construction of the same dispatch: a stable sort of (expert, slot).

    Used only to pin `permute` against itself-by-another-route in the tests.
    """
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")          # slots grouped by expert, slot order kept
    counts = np.bincount(flat, minlength=E)
    starts = np.concatenate([[0], np.cumsum(counts)])
    rank = np.empty(T * k, dtype=np.int64)           # rank of each slot inside its expert
    rank[order] = np.arange(T * k) - starts[flat[order]]
    keep = np.ones(T * k, dtype=bool) if C is None else rank < C
    kept = np.bincount(flat[keep], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(kept)])
    slot_pos = np.where(keep, offsets[flat] + rank, -1)
    perm_slot = np.full(T * k, -1, dtype=np.int64)
    perm_slot[slot_pos[keep]] = np.nonzero(keep)[0]
    return {"counts": counts.astype(np.int32), "offsets": offsets.astype(np.int32),
            "perm_slot": perm_slot.astype(np.int32), "slot_pos": slot_pos.astype(np.int32),
            "n_kept": int(offsets[E])}


# ----------------------------------------------------------------------------------------
# experts and combine
# ----------------------------------------------------------------------------------------
def overflow_reroute(topk_idx, slot_pos, scores, E: int, C: int):
    """Level-2 capacity protection ("参数规模与稀疏激活的真相拆解", §3.2 专家容量: overflow tokens
    are not dropped but handed to a fallback router that picks the next-best expert that is not
    full). Reading where the page is silent: after the Level-1 walk (`permute`), the dropped
    slots are visited in slot order (t ascending, then j); each takes the expert with the best
    selection score (ties to the lower index) among those that still have room and that its token
    does not already use; the slot stays dropped when there is none. Each taken expert's room
    shrinks by one before the next dropped slot is visited.

    Returns dict(topk_idx [T, k] with the re-routed experts in place, rerouted [T, k] bool,
    margin [T]: the smallest gap, over the token's re-routed slots, between the chosen score and
    the best other eligible score (inf when none))."""
    idx = np.array(topk_idx, np.int64)
    T, k = idx.shape
    s = np.asarray(scores, np.float64)
    sp = np.asarray(slot_pos, np.int64)
    fill = np.zeros(E, np.int64)
    for t in range(T):
        for j in range(k):
            if sp[t * k + j] >= 0:
                fill[idx[t, j]] += 1
    out = idx.copy()
    rerouted = np.zeros((T, k), bool)
    margin = np.full(T, np.inf)
    for t in range(T):
        used = {int(idx[t, j]) for j in range(k) if sp[t * k + j] >= 0}
        for j in range(k):
            if sp[t * k + j] >= 0:
                continue
            elig = sorted((e for e in range(E) if fill[e] < C and e not in used),
                          key=lambda e: (-s[t, e], e))
            if not elig:
                continue
            best = elig[0]
            if len(elig) > 1:
                a, b = s[t, best], s[t, elig[1]]
                margin[t] = min(margin[t], a - b if a != b else 0.0)
            out[t, j] = best
            rerouted[t, j] = True
            fill[best] += 1
            used.add(best)
    return {"topk_idx": out.astype(np.int32), "rerouted": rerouted, "margin": margin}


def overflow_reroute_by_proposals(topk_idx, slot_pos, scores, E: int, C: int):
    """Second, independent construction of `overflow_reroute`, used only to pin it: every token
    with dropped slots proposes to its best untried experts (one per unmet slot); each expert
    keeps the proposals of the lowest-numbered tokens up to its room and turns the others away;
    turned-away tokens propose again, until no proposal is turned away. With one priority order
    (token number) shared by all experts this ends in the same assignment as the slot-order walk.
    Returns the final topk_idx."""
    idx = np.array(topk_idx, np.int64)
    T, k = idx.shape
    s = np.asarray(scores, np.float64)
    sp = np.asarray(slot_pos, np.int64).reshape(T, k)
    room = np.full(E, C, np.int64)
    for t in range(T):
        for j in range(k):
            if sp[t, j] >= 0:
                room[idx[t, j]] -= 1
    want = {t: int((sp[t] < 0).sum()) for t in range(T) if (sp[t] < 0).any()}
    pref = {t: [e for e in sorted(range(E), key=lambda e: (-s[t, e], e))
                if e not in {int(idx[t, j]) for j in range(k) if sp[t, j] >= 0}] for t in want}
    nxt = {t: 0 for t in want}
    held = {e: set() for e in range(E)}
    while True:
        for t in want:
            have = sum(t in held[e] for e in range(E))
            while have < want[t] and nxt[t] < len(pref[t]):
                held[pref[t][nxt[t]]].add(t)
                nxt[t] += 1
                have += 1
        turned = False
        for e in range(E):
            if len(held[e]) > room[e]:
                keep = sorted(held[e])[:max(room[e], 0)]
                turned = True
                held[e] = set(keep)
        if not turned:
            break
    out = idx.copy()
    for t in want:
        got = sorted((e for e in range(E) if t in held[e]), key=lambda e: (-s[t, e], e))
        for j, e in zip([j for j in range(k) if sp[t, j] < 0], got):
            out[t, j] = e
    return out.astype(np.int32)


def silu(z):
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(xrows, W_gate, W_up, W_down) -> np.ndarray:
    """y = (silu(x W_gate) * (x W_up)) W_down for a block of rows, no intermediate rounding."""
    xr = np.asarray(xrows, np.float64)
    g = xr @ np.asarray(W_gate, np.float64)
    u = xr @ np.asarray(W_up, np.float64)
    return (silu(g) * u) @ np.asarray(W_down, np.float64)


def combine(T, k, d, topk_w, slot_pos, slot_y, shared_y=None, tokens=None):
    """out[t] = sum over kept j of topk_w[t,j] * y(t,j)  +  sum over shared s of z_s[t].

    slot_y: dict slot -> y row (unscaled expert output) for every kept slot of the tokens asked.
    shared_y: list over shared experts of dict t -> z row (or None).
    Returns float64 [len(tokens), d].
    """
    toks = range(T) if tokens is None else tokens
    out = np.zeros((len(toks), d), dtype=np.float64)
    for r, t in enumerate(toks):
        for j in range(k):
            slot = t * k + j
            if slot_pos[slot] >= 0:
                out[r] += topk_w[t, j] * slot_y[slot]
        if shared_y is not None:
            for zs in shared_y:
                out[r] += zs[t]
    return out


def expert_outputs(x, topk_idx, slot_pos, get_expert, k, tokens=None, n_shared=0,
                   get_shared=None):
    """Run each expert on the kept slots of the requested tokens.

    get_expert(e) -> (W_gate [d,f], W_up [d,f], W_down [f,d]) as float64 (or bf16-exact) arrays;
    weights are fetched one expert at a time so that large layers never need every expert in
    float64 at once.  Returns (slot_y dict, shared_y list of dicts).
    """
    idx = np.asarray(topk_idx, np.int64)
    T = idx.shape[0]
    toks = list(range(T)) if tokens is None else list(tokens)
    by_expert: dict[int, list[int]] = {}
    for t in toks:
        for j in range(k):
            slot = t * k + j
            if slot_pos[slot] >= 0:
                by_expert.setdefault(int(idx[t, j]), []).append(slot)
    slot_y = {}
    for e in sorted(by_expert):
        slots = by_expert[e]
        Wg, Wu, Wd = get_expert(e)
        y = swiglu_expert(np.asarray(x)[[s // k for s in slots]], Wg, Wu, Wd)
        for i, s in enumerate(slots):
            slot_y[s] = y[i]
    shared_y = []
    for s_i in range(n_shared):
        Wg, Wu, Wd = get_shared(s_i)
        z = swiglu_expert(np.asarray(x)[toks], Wg, Wu, Wd)
        shared_y.append({t: z[r] for r, t in enumerate(toks)})
    return slot_y, shared_y


def layer_from_routing(x, topk_idx, topk_w, E, C, get_expert, n_shared=0, get_shared=None,
                       tokens=None):
    """Permute + experts + combine on given routing decisions (the conditioned oracle)."""
    x = np.asarray(x, np.float64)
    T, d = x.shape
    k = np.asarray(topk_idx).shape[1]
    perm = permute(topk_idx, E, C)
    slot_y, shared_y = expert_outputs(x, topk_idx, perm["slot_pos"], get_expert, k,
                                      tokens, n_shared, get_shared)
    out = combine(T, k, d, np.asarray(topk_w, np.float64), perm["slot_pos"], slot_y,
                  shared_y if n_shared else None, tokens)
    return out, perm


def layer(x, W_g, k, get_expert, E, mode=PLAIN, expert_bias=None, gumbel_u=None, tau=1.0,
          capacity_factor=0.0, capacity_override=0, n_shared=0, get_shared=None, tokens=None,
          n_groups=0, topk_groups=0, reroute=False):
    """The whole layer: route -> permute (with capacity) -> SwiGLU experts -> combine.

    `tokens` restricts the expert and combine work to those tokens (routing and the capacity
    walk always run over every token, since a token's keep/drop status depends on earlier ones).
    Returns dict(out f64 [len(tokens), d], route dict, perm dict, C).
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    r = route(x, W_g, k, mode, expert_bias, gumbel_u, tau, n_groups, topk_groups)
    C = capacity(T, k, E, capacity_factor, capacity_override)
    idx, w = r["topk_idx"], r["topk_w"]
    if reroute and C is not None:
        # Level 2: dropped slots move to the best expert with room; gates over the final experts
        rr = overflow_reroute(idx, permute(idx, E, C)["slot_pos"], r["scores"], E, C)
        idx = rr["topk_idx"]
        w = gates(r["logits"], r["scores"], idx, mode)
        r = dict(r, reroute=rr)
    out, perm = layer_from_routing(x, idx, w, E, C, get_expert, n_shared, get_shared, tokens)
    return {"out": out, "route": r, "perm": perm, "C": C, "topk_idx": idx, "topk_w": w}


def layer_dense(x, W_g, k, experts, mode=PLAIN, expert_bias=None, gumbel_u=None, tau=1.0,
                shared=()):
    """Every expert on every token, then masked by the routing and weighted: a second route to
    the same layer output (no capacity), sharing no dispatch code with `layer`.

    experts: list of (W_gate, W_up, W_down); shared: list of the same for shared experts.
    """
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = len(experts)
    r = route(x, W_g, k, mode, expert_bias, gumbel_u, tau)
    gate_full = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            gate_full[t, r["topk_idx"][t, j]] = r["topk_w"][t, j]
    out = np.zeros((T, np.asarray(experts[0][2]).shape[1]))
    for e, (Wg, Wu, Wd) in enumerate(experts):
        out += gate_full[:, e:e + 1] * swiglu_expert(x, Wg, Wu, Wd)
    for (Wg, Wu, Wd) in shared:
        out += swiglu_expert(x, Wg, Wu, Wd)
    return out


# ----------------------------------------------------------------------------------------
# next rows (after the forward pass)
# ----------------------------------------------------------------------------------------
def bias_update(expert_bias, counts, decay=0.99, rate=0.01, eps=1e-8):
    """Aux-loss-free bias update after a forward pass
    ("AI架构演进从稀疏MoE到条件记忆的工程实践", gating-network code, its no_grad block):
      load = per-expert slot counts (all k picks, before any capacity limit)
      bias <- decay * bias - rate * load / (mean(load) + eps)
    """
    b = np.asarray(expert_bias, np.float64)
    load = np.asarray(counts, np.float64)
    return decay * b - rate * load / (load.mean() + eps)


# ----------------------------------------------------------------------------------------
# weight-only group-wise quantized experts
# ----------------------------------------------------------------------------------------
QUANT_GROUP = 128


def quantize_groupwise(W, bits: int, group: int = QUANT_GROUP):
    """Group-wise asymmetric weight quantization ("大模型MoE稀疏激活原理与工程实践", §4.2
    量化与混合精度: expert weights to INT4, one scale and zero-point per group of 128 weights;
    the block quantizer of "GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token",
    §4 INT4 block quantization: scale = (max - min) / 15 kept in FP16, zero_point =
    round(-min / scale)). Readings where the pages are silent: a group is 128 consecutive
    weights along the input (reduction) dimension of one output column; b-bit codes are
    unsigned, q = clamp(rint(w / s) + z, 0, 2^b - 1), w' = (q - z) * s; s is rounded to fp16
    (a zero or non-finite s becomes fp16(max |w|), or 1 for an all-zero group); z = clamp(
    rint(-min / s), 0, 2^b - 1); every division is in float64; rint rounds half to even.

    W: [..., K, N] float (the bf16 weights widened); returns (q uint8 [..., K, N],
    s float16 [..., K / group, N], z uint8 [..., K / group, N])."""
    W = np.asarray(W, np.float64)
    *lead, K, N = W.shape
    assert K % group == 0
    top = float(2 ** bits - 1)
    Wg = W.reshape(*lead, K // group, group, N)
    lo = Wg.min(axis=-2)
    hi = Wg.max(axis=-2)
    s = ((hi - lo) / top).astype(np.float16)
    bad = (s == 0) | ~np.isfinite(s)
    if bad.any():
        alt = np.maximum(np.abs(lo), np.abs(hi)).astype(np.float16)
        alt = np.where((alt == 0) | ~np.isfinite(alt), np.float16(1.0), alt)
        s = np.where(bad, alt, s)
    s64 = s.astype(np.float64)
    z = np.clip(np.rint(-lo / s64), 0, top)
    q = np.clip(np.rint(Wg / s64[..., None, :]) + z[..., None, :], 0, top)
    return (q.reshape(*lead, K, N).astype(np.uint8), s, z.astype(np.uint8))


def dequantize_groupwise(q, s, z, group: int = QUANT_GROUP):
    """w' = (q - z) * s per group (exact in float64)."""
    q = np.asarray(q, np.float64)
    *lead, K, N = q.shape
    sg = np.repeat(np.asarray(s, np.float64), group, axis=-2)
    zg = np.repeat(np.asarray(z, np.float64), group, axis=-2)
    return (q - zg) * sg
