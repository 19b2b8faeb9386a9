"""CPU oracle of the routed INT4-expert MoE FFN -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package's smoke check and the benchmark's CPU-baseline
leg may import this module. The library and its Python binding never do: the
product path runs in the CUDA library and fails loudly without it.

Plain, slow and written to be checked by eye. Floating point is FP64 (numpy
float64); inputs arrive in the precisions the pages fix (FP16 activations and
scales, packed INT4 codes, FP32 router logits) and are widened exactly. The
only library primitives used are numpy's matrix product, exp/log and sorting.

Sources (web pages; cited by title and section):
* "Horizon RunMap -- Prévia Técnica" (horizonrunmap.com/pt), sections
  "02 / A solução", "03 / Arquitetura" (the resident-qpacked-cache-v1 /
  ADR 0009 contract) and "08 / Comportamento do modelo" (W4A16: INT4 expert
  weights, FP16 scales, FP16 activations, FP32 accumulation).
* "Horizon RunMap claims.json", experiment ``contract`` (canonical initial
  placement; one decode step at a time).
* "Desenvolvedor do Strata cria mapa ao vivo de 24 576 especialistas MoE em
  uma GTX 1070", section "Como 125 bilhões de parâmetros cabem em 8 GB"
  (eviction by an access counter whose old accesses lose weight).
* lucashiago.com.br "local" explainer, etapa 1 (a scale and a zero point per
  block of weights), etapa 3 (experts touched by n tokens), etapa 4 (the hit
  ceiling of any cache policy; profile against LRU), etapa 5 (the declared
  time model t = t_calc + bytes_out / bandwidth).
* "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura", ADR 0009: copies
  land in spare positions before a generation is published (prefetch into
  spare slots).

Readings where the pages are silent (listed with reasons in the design notes):
groups run along each row's reduction axis; code element 2c is the low nibble
of byte c; w = (q - z) * s; top-k on raw logits ordered by (logit desc, index
asc); softmax over all E logits, optionally renormalised over the chosen k;
SwiGLU expert h = silu(W_g x) * (W_u x), o = W_d h; y = sum_j w_j o_j plus the
shared path's output; the decayed-count policy steps below.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Storage: packed 4-bit codes, per-group FP16 scale and zero point.
# "08 / Comportamento do modelo": expert weights INT4, scales FP16, converted
# inside the kernel. lucashiago etapa 1: every block of weights carries the
# scale and the zero point that rebuild it.
# --------------------------------------------------------------------------
def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[rows][cols/2] bytes -> [rows][cols] integer codes 0..15.

    Element 2c is the low nibble of byte c, element 2c+1 the high nibble.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    q = np.empty((rows, 2 * half), dtype=np.int64)
    q[:, 0::2] = packed & 0x0F
    q[:, 1::2] = packed >> 4
    return q


def dequantize(packed: np.ndarray, scale: np.ndarray, zero: np.ndarray,
               group: int) -> np.ndarray:
    """W[n][c] = (q[n][c] - z[n][c // g]) * s[n][c // g], in float64."""
    q = unpack_codes(packed)
    rows, cols = q.shape
    s = np.asarray(scale, dtype=np.float64)
    z = np.asarray(zero, dtype=np.float64)
    assert cols % group == 0 and s.shape == (rows, cols // group) == z.shape
    gi = np.arange(cols) // group  # the group of every column c
    return (q - z[:, gi]) * s[:, gi]


def dequantize_expert(arrs: dict, group: int) -> tuple:
    """(W_g [I][H], W_u [I][H], W_d [H][I]) of one expert, float64."""
    wg = dequantize(arrs["qp_gate"], arrs["s_gate"], arrs["z_gate"], group)
    wu = dequantize(arrs["qp_up"], arrs["s_up"], arrs["z_up"], group)
    wd = dequantize(arrs["qp_down"], arrs["s_down"], arrs["z_down"], group)
    return wg, wu, wd


# --------------------------------------------------------------------------
# Router. "02 / A solução" and "03 / Arquitetura": the router picks, for each
# token and routed layer, the experts that work on it; it stays outside INT4.
# --------------------------------------------------------------------------
class NonFiniteLogits(ValueError):
    pass


def route(logits: np.ndarray, k: int, renorm: bool) -> tuple:
    """Top-k experts per token and their weights.

    Selection: experts ordered by (logit descending, index ascending); the
    first k are chosen, in that order. Weights: p = softmax over all E logits
    in float64; w_j = p[id_j] / sum_j' p[id_j'] when ``renorm``, else p[id_j].
    NaN or +inf logits, or a token with every logit -inf, are rejected.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("k must be in [1, E]")
    ids = np.zeros((T, k), dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        row = logits[t]
        if np.any(np.isnan(row)) or np.any(row == np.inf) or np.all(row == -np.inf):
            raise NonFiniteLogits(f"token {t}")
        order = sorted(range(E), key=lambda e: (-float(row[e]), e))
        chosen = order[:k]
        l64 = row.astype(np.float64)
        m = float(np.max(l64))
        p = np.exp(l64 - m)
        p = p / np.sum(p)
        pw = np.array([p[e] for e in chosen])
        if renorm:
            pw = pw / np.sum(pw)
        ids[t] = chosen
        w[t] = pw
    return ids, w


# --------------------------------------------------------------------------
# Expert FFN (SwiGLU) and the weighted combine.
# "03 / Arquitetura": the expert kernel takes the FP16 activations and returns
# its result to the rest of the model; the router's choice weighs it.
# --------------------------------------------------------------------------
def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def expert_ffn(x: np.ndarray, wg: np.ndarray, wu: np.ndarray,
               wd: np.ndarray) -> np.ndarray:
    """o = W_d (silu(W_g x) * (W_u x)) for one token x [H], float64."""
    x = np.asarray(x, dtype=np.float64)
    g = wg @ x
    u = wu @ x
    h = silu(g) * u
    return wd @ h


def moe_layer(x: np.ndarray, logits: np.ndarray, experts, k: int,
              renorm: bool, group: int, y_shared=None) -> dict:
    """One routed layer: y[t] = sum_j w[t][j] * o(x[t]; expert ids[t][j]) (+ y_shared[t]).

    ``experts`` maps an expert id to its canonical arrays (a dict or a
    callable). Only the touched experts are dequantised, once each.
    Returns {"y": float64 [T][H], "ids", "weights"}.
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    T, H = x.shape
    ids, w = route(logits, k, renorm)
    cache = {}

    def mats(e):
        if e not in cache:
            arrs = experts(e) if callable(experts) else experts[e]
            cache[e] = dequantize_expert(arrs, group)
        return cache[e]

    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            wg, wu, wd = mats(int(ids[t, j]))
            y[t] += w[t, j] * expert_ffn(x[t], wg, wu, wd)
    if y_shared is not None:
        y += np.asarray(y_shared, dtype=np.float64)
    return {"y": y, "ids": ids, "weights": w}


def moe_layer_dense(x: np.ndarray, logits: np.ndarray, experts, E: int, k: int,
                    renorm: bool, group: int) -> np.ndarray:
    """Brute force: run every expert on every token, then mask by the routing.

    G[t][e] = w[t][j] if e == ids[t][j] else 0; y[t] = sum_e G[t][e] o_e(x[t]).
    An independent second evaluation of the routed layer.
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    T, H = x.shape
    ids, w = route(logits, k, renorm)
    gate = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            gate[t, ids[t, j]] = w[t, j]
    y = np.zeros((T, H), dtype=np.float64)
    for e in range(E):
        arrs = experts(e) if callable(experts) else experts[e]
        wg, wu, wd = dequantize_expert(arrs, group)
        o = np.stack([expert_ffn(x[t], wg, wu, wd) for t in range(T)])
        y += gate[:, e:e + 1] * o
    return y


# --------------------------------------------------------------------------
# Non-routed FP16 path. "03 / Arquitetura": the parts outside the routed
# experts run in FP16; "08 / Comportamento do modelo": the non-routed weights
# are FP16. Same SwiGLU form with FP16 weights widened exactly.
# --------------------------------------------------------------------------
def shared_ffn(x: np.ndarray, wg: np.ndarray, wu: np.ndarray,
               wd: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    g = x @ np.asarray(wg, dtype=np.float64).T
    u = x @ np.asarray(wu, dtype=np.float64).T
    h = silu(g) * u
    return h @ np.asarray(wd, dtype=np.float64).T


# --------------------------------------------------------------------------
# Token sort for the grouped executor ("04 / Resultados": compact experts
# computed in groups). Pairs p = t*k + j ordered by (expert, p).
# --------------------------------------------------------------------------
def token_sort(ids: np.ndarray, E: int) -> tuple:
    """Returns (offsets [E+1], pair_tok [T*k], pair_j [T*k])."""
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = [int(v) for v in ids.reshape(-1)]
    order = sorted(range(T * k), key=lambda p: (flat[p], p))
    counts = [0] * E
    for e in flat:
        counts[e] += 1
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    pair_tok = np.array([p // k for p in order], dtype=np.int32)
    pair_j = np.array([p % k for p in order], dtype=np.int32)
    return np.array(offsets, dtype=np.int32), pair_tok, pair_j


# --------------------------------------------------------------------------
# Residency policy: decayed access counts (Strata page), a fixed per-layer
# capacity declared before requests and canonical initial placement
# ("03 / Arquitetura" ADR 0009 list; claims.json ``contract``).
# --------------------------------------------------------------------------
class CapacityError(ValueError):
    pass


class ResidencyLayer:
    """Decision model of one layer's GPU slot pool.

    C experts may be resident; the pool has C + S physical slots (S spares).
    Start: expert e in slot e for e < C, counts 0, slots C.. free.
    One step with the ids needed by all tokens of this decode step:
      1. every count c becomes c * decay, then gains 1.0 per occurrence;
      2. N = the distinct needed ids; |N| > C is a capacity error;
      3. misses N \\ R in ascending id order; for each, if |R| = C a victim
         leaves R; the miss takes the lowest free slot, else the victim's slot;
      4. slots of victims that were not reused become free after the step.
    Victims, over R \\ N:
      "decay"  (Strata page: an access counter whose old accesses lose
               weight): argmin of (count_v, v);
      "lru"    (claims.json experiment contract: evolving LRU): argmin of
               (last step v was needed, v), never needed = -1;
      "pinned" (lucashiago.com.br "local", etapa 4: a measured profile pins
               the popular set): the `pinned` experts with the largest
               profile value (ties: lower id) are never victims and are
               resident from the start together with the lowest other ids
               (slots in ascending id order); the others follow "lru".
    Prefetch ("03 / Arquitetura", ADR 0009: a copy lands in a spare
    position before it is published): prefetch(ids) stages each listed
    expert that is neither resident nor staged into the lowest free slot,
    while one is free; the next step takes a staged expert it needs as a
    miss in its staged slot (victim chosen as usual, the victim's slot then
    goes free), and returns the staged experts it does not need to the free
    slots.
    """

    def __init__(self, E: int, C: int, S: int, decay: float, policy: str = "decay",
                 profile=None, pinned: int = 0):
        if not (1 <= C <= E) or S < 0:
            raise CapacityError("bad capacity")
        if policy not in ("decay", "lru", "pinned"):
            raise ValueError("unknown policy")
        self.E, self.C, self.S, self.decay = E, C, S, float(decay)
        self.policy = policy
        self.counts = [0.0] * E
        self.last_used = [-1] * E
        self.steps = 0
        self.pinned = set()
        self.slot_of = [-1] * E
        if policy == "pinned":
            order = sorted(range(E), key=lambda e: (-float(profile[e]), e))
            self.pinned = set(order[:pinned])
            resident = set(self.pinned)
            for e in range(E):
                if len(resident) >= C:
                    break
                resident.add(e)
            for slot, e in enumerate(sorted(resident)):
                self.slot_of[e] = slot
        else:
            for e in range(C):
                self.slot_of[e] = e
        self.free = list(range(C, C + S))
        self.staged = {}  # expert -> slot holding its prefetched copy
        self.hits = self.misses = self.evictions = 0
        self.prefetched = self.prefetch_copies = 0

    def prefetch(self, ids) -> list:
        """Stage predicted misses; returns [(expert, slot)] in staging order."""
        ids = [int(e) for e in ids]
        if any(e < 0 or e >= self.E for e in ids):
            raise ValueError("expert id out of range")
        out = []
        for e in ids:
            if not self.free:
                break
            if self.slot_of[e] >= 0 or e in self.staged:
                continue
            slot = min(self.free)
            self.free.remove(slot)
            self.staged[e] = slot
            out.append((e, slot))
        self.prefetch_copies += len(out)
        return out

    def resident(self):
        return [e for e in range(self.E) if self.slot_of[e] >= 0]

    def step(self, needed) -> list:
        """Apply one step; returns [(expert, slot, victim or -1)] per miss."""
        needed = [int(e) for e in needed]
        if any(e < 0 or e >= self.E for e in needed):
            raise ValueError("expert id out of range")
        distinct = sorted(set(needed))
        if len(distinct) > self.C:
            raise CapacityError("more distinct experts than slots")
        for e in range(self.E):
            self.counts[e] = self.counts[e] * self.decay
        for e in needed:
            self.counts[e] = self.counts[e] + 1.0
        resident = set(self.resident())
        misses = [e for e in distinct if e not in resident]
        self.hits += len(distinct) - len(misses)
        self.misses += len(misses)
        decisions = []
        retiring = []
        for e in misses:
            victim = -1
            if len(resident) == self.C:
                candidates = [v for v in resident if v not in distinct and v not in self.pinned]
                if self.policy == "decay":
                    victim = min(candidates, key=lambda v: (self.counts[v], v))
                else:
                    victim = min(candidates, key=lambda v: (self.last_used[v], v))
                resident.remove(victim)
                retiring.append(self.slot_of[victim])
                self.slot_of[victim] = -1
                self.evictions += 1
            if e in self.staged:
                slot = self.staged[e]
                self.prefetched += 1
            elif self.free:
                slot = min(self.free)
                self.free.remove(slot)
            else:
                slot = retiring.pop()
            self.slot_of[e] = slot
            resident.add(e)
            decisions.append((e, slot, victim))
        self.free.extend(retiring)
        self.free.extend(slot for e, slot in self.staged.items() if e not in distinct)
        self.staged = {}
        for e in distinct:
            self.last_used[e] = self.steps
        self.steps += 1
        return decisions


def residency_sim(id_steps, E: int, C: int, S: int, decay: float, policy: str = "decay",
                  profile=None, pinned: int = 0) -> dict:
    """Run the policy of one layer over a sequence of steps (lists of ids)."""
    layer = ResidencyLayer(E, C, S, decay, policy, profile, pinned)
    trace = []
    for step, needed in enumerate(id_steps):
        for (e, slot, victim) in layer.step(needed):
            trace.append((step, e, slot, victim))
    return {"trace": trace, "hits": layer.hits, "misses": layer.misses,
            "evictions": layer.evictions, "slot_of": list(layer.slot_of),
            "counts": list(layer.counts)}


# --------------------------------------------------------------------------
# Closed forms from the lucashiago explainer (etapas 3 and 4).
# --------------------------------------------------------------------------
def expected_touched(E: int, k: int, n: int) -> float:
    """Mean number of distinct experts n independent tokens touch: E(1-(1-k/E)^n)."""
    return E * (1.0 - (1.0 - k / E) ** n)


def hit_ceiling(p, C: int) -> float:
    """Best possible hit rate: the sum of the C largest access probabilities."""
    return float(sum(sorted(p, reverse=True)[:C]))


def expert_block_bytes(H: int, I: int, g: int) -> int:
    """Bytes of one expert: 3*H*I/2 code bytes + FP16 scale and zero per group."""
    return 3 * H * I // 2 + 3 * (H * I // g) * 2 * 2


# --------------------------------------------------------------------------
# Cost of weights outside the fast memory (lucashiago explainer, etapa 5):
# every weight not resident is read again at each use, and the declared
# model prices a unit of work as t = t_calc + bytes_out / bandwidth, with no
# overlap between the reads and the computation.
# --------------------------------------------------------------------------
def time_model(t_calc: float, bytes_out: float, bandwidth: float) -> float:
    """Time of one unit of work whose non-resident weights total bytes_out.

    The model is additive over tokens, so a unit may be one token or a whole
    response (its summed compute time and summed traffic)."""
    return t_calc + bytes_out / bandwidth


def fit_time_model(bytes_out, times) -> tuple:
    """(t_calc, bandwidth) of time_model by least squares over measured
    (bytes_out, time) points: numpy lstsq on the columns [1, bytes_out]."""
    b = np.asarray(bytes_out, dtype=np.float64)
    t = np.asarray(times, dtype=np.float64)
    A = np.stack([np.ones_like(b), b], axis=1)
    (t_calc, per_byte), *_ = np.linalg.lstsq(A, t, rcond=None)
    return float(t_calc), float(1.0 / per_byte)


def expected_outside(E: int, C: int, k: int, n: int) -> float:
    """Mean number of distinct non-resident experts that n tokens touch when
    C of the E experts are resident and each token picks a uniform random
    k-subset (etapa 3's per-expert miss probability (1-k/E)^n, applied to
    each of the E - C experts outside)."""
    return (E - C) * (1.0 - (1.0 - k / E) ** n)
