"""Autoregressive decoding, depth exploration decoding (DEX), depth-coupled sampling
(DECS) and brute-force EAD -- oracle side.

Written from the prose of "Depth Exploration for LLM Decoding" (arXiv 2606.29223),
section 3.2 (lattice expansion, commit, finite-state control and collapse) and
section 3.3 / Appendix C.1 (depth-coupled sampling), with the readings below where
the pages leave a step open.  TEST INFRASTRUCTURE ONLY.

Lattice (section 3.2, Figure 2).  Exploration tokens ETK_i live in a binary tree in
heap order: the root ETK_0 is the stage-0 node of the commit position p_c; node i has a
depth child D(i) = 2i+1 (same token position, next explorer) and a position child
P(i) = 2i+2 (its candidate becomes the next position's token, restart at explorer 0).
This matches "ETK_1 in the same slot chain, ETK_2 the first token of a new slot" and
"state q materializes the first 2^q - 1 tokens".  The round at state q computes the
2^q nodes of level q; the anchor path is D^k(0) = 2^k - 1, k = 0..N-1.

Node semantics.  A node is the model evaluated on its token prefix: the committed
tokens followed by the candidates of the P-parents on its path; its stage s is the
number of trailing depth moves, and its candidate comes from the shared exit head at
depth d_s (Appendix C.2), decoded by DECS.

Readings taken where the pages are silent:
* q after collapse = N - k* - 1: the survivors are the subtree of the new anchor
  m = P(b_{k*}) = 2^(k*+1), created k*+1 rounds into the cycle, re-indexed
  i -> i - m * 2^h (h = depth of i below m); fallback k* = N-1 leaves nothing, q = 0.
* DECS masks Prior(i) = the tokens of the shallower nodes of i's slot chain, except
  at the final-depth reference (stage N-1, which only the anchor reaches).
* Sampling draws the Gumbel row of the node's absolute target position (see philox).
* Greedy argmax breaks ties toward the lowest token id.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import analysis
from .philox import gumbel_row


# -------------------------------------------------------------------------------------
# lattice indexing
# -------------------------------------------------------------------------------------

def parent(i: int) -> int:
    return (i - 1) // 2


def depth_child(i: int) -> int:
    return 2 * i + 1


def position_child(i: int) -> int:
    return 2 * i + 2


def is_depth_child(i: int) -> bool:
    return i > 0 and i % 2 == 1


def level(i: int) -> int:
    return (i + 1).bit_length() - 1


def level_nodes(q: int) -> range:
    """The 2^q nodes created by the round at state q."""
    return range(2 ** q - 1, 2 ** (q + 1) - 1)


def stage(i: int) -> int:
    """Explorer index of node i: number of trailing depth moves on its path."""
    s = 0
    while is_depth_child(i):
        s += 1
        i = parent(i)
    return s


def slot_root(i: int) -> int:
    """r(i): first node of i's slot chain (the root or a position child)."""
    while is_depth_child(i):
        i = parent(i)
    return i


def prior_nodes(i: int) -> List[int]:
    """Prior(i): shallower nodes of the same slot chain (Appendix C.1)."""
    out = []
    while is_depth_child(i):
        i = parent(i)
        out.append(i)
    return out


def branch_parents(i: int) -> List[int]:
    """Nodes whose candidates extend i's prefix (the P-parents on the root->i path), root first."""
    out = []
    while i > 0:
        p = parent(i)
        if i % 2 == 0:
            out.append(p)
        i = p
    return out[::-1]


def anchor_node(k: int) -> int:
    """b_k = D^k(0), the anchor-path node at explorer k."""
    return 2 ** k - 1


def subtree_remap(m: int, max_level: int) -> Dict[int, int]:
    """Old -> new heap index for the subtree of m restricted to levels <= max_level.

    Closed form of the collapse re-indexing: i -> i - m * 2^h, h = level(i) - level(m).
    """
    out = {}
    frontier = [m]
    while frontier:
        nxt = []
        for i in frontier:
            if level(i) > max_level:
                continue
            h = level(i) - level(m)
            out[i] = i - m * 2 ** h
            nxt += [depth_child(i), position_child(i)]
        frontier = nxt
    return out


# -------------------------------------------------------------------------------------
# decoding rule and DECS
# -------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Rule:
    """Final-depth decoding rule R: greedy, or Gumbel-max sampling at temperature tau."""
    sample: bool = False
    tau: float = 1.0
    seed: int = 0


def first_argmax(score: np.ndarray) -> int:
    """argmax with ties broken toward the lowest index."""
    return int(np.flatnonzero(score == score.max())[0])


def decision_scores(logits: np.ndarray, rule: Rule, seq: int, target_pos: int) -> np.ndarray:
    """The scores whose argmax is the token: logits (greedy) or logits / tau + G (sampling)."""
    if not rule.sample:
        return logits
    return logits / rule.tau + gumbel_row(rule.seed, seq, target_pos, logits.shape[-1])


def margin(score: np.ndarray) -> float:
    """Top-1 minus top-2 of the decision scores (ignoring masked -inf entries)."""
    finite = np.sort(score[np.isfinite(score)])
    return float(finite[-1] - finite[-2]) if finite.size >= 2 else float("inf")


def depth_coupled_token(logits: np.ndarray, shallower: Sequence[int], final_depth: bool, rule: Rule,
                        seq: int, target_pos: int, enabled: bool = True) -> Tuple[int, float, List[int]]:
    """One exploration token of a slot chain under depth-coupled sampling (section 3.3;
    Appendix C.1).

    ``shallower`` holds the tokens the chain already proposed at shallower depths.  They
    are excluded from this depth's choice -- a repeat could never add a new match -- except
    for the final-depth reference, which always sees the unmasked logits so the committed
    token is exactly the decoding rule's token.  With ``enabled=False`` nothing is excluded
    (the independent "vanilla" decoding of the section 4.1 ablation).

    Returns (token, margin of the decision scores, excluded token ids).
    """
    excluded = sorted(set(int(v) for v in shallower)) if (enabled and not final_depth) else []
    z = np.array(logits, dtype=np.float64, copy=True)
    if excluded:
        z[excluded] = -np.inf
    score = decision_scores(z, rule, seq, target_pos)
    return first_argmax(score), margin(score), excluded


# -------------------------------------------------------------------------------------
# autoregressive decoding (the lossless target) and brute-force EAD
# -------------------------------------------------------------------------------------

@dataclass
class ARResult:
    tokens: List[int]
    logits: List[np.ndarray]                       # final-depth logits per generated token
    margins: List[float]
    depth_candidates: Optional[List[List[int]]] = None   # [t][l-1]: candidate at depth l


def prefill(model, prompt: Sequence[int], capacity: int):
    """The committed context of a prompt: a cache of ``capacity`` positions holding the KV
    state of positions 0..P-2.  The last prompt token is the first decode step's input, so
    its position is computed by the decode itself (section 2.1 / 3.2 alike).

    A decode started from this cache writes only positions >= P-1, so the same prefilled
    cache serves any number of decodes of the same prompt."""
    cache = model.new_cache(capacity)
    if len(prompt) > 1:
        model.forward([int(t) for t in prompt[:-1]], 0, cache)
    return cache


def ar_generate(model, prompt: Sequence[int], T: int, rule: Rule = Rule(), seq: int = 0,
                record_depths: bool = False, force: Optional[Sequence[int]] = None, cache=None) -> ARResult:
    """Standard AR decoding of T tokens (section 2.1): every token through all L layers.

    Prompt positions 0..P-2 are prefilled (or taken from ``cache``, a ``prefill`` of the same
    prompt with room for P + T + 1 positions); the last prompt token at position P-1 yields
    the first new token (position P).  With ``force`` the given tokens are appended instead of
    the decoded ones (teacher forcing: scores a token stream produced elsewhere).  With
    ``record_depths`` the candidate of every depth l in [L] under the same rule is kept.
    """
    P = len(prompt)
    if cache is None:
        cache = prefill(model, prompt, P + T + 1)
    last, pos = int(prompt[-1]), P - 1
    out = ARResult([], [], [], [] if record_depths else None)
    for t in range(T):
        hist = model.forward([last], pos, cache, keep_depths=True)
        z = model.exit_logits(hist[-1])[0]
        score = decision_scores(z, rule, seq, pos + 1)
        y = first_argmax(score)
        out.logits.append(z)
        out.margins.append(margin(score))
        if record_depths:
            cands = []
            for l in range(model.L):
                zl = model.exit_logits(hist[l])[0]
                cands.append(first_argmax(decision_scores(zl, rule, seq, pos + 1)))
            out.depth_candidates.append(cands)
        if force is not None:
            y = int(force[t])
        out.tokens.append(y)
        last, pos = y, pos + 1
    return out


def ead_profile(ar: ARResult):
    """Brute-force Def. 1: Omega(t, l) = [candidate at depth l == final-depth token].

    Returns (omega rows, EAD(t) list, stable EAD(t) list).
    """
    omegas, eads, stabs = [], [], []
    for t, y in enumerate(ar.tokens):
        omega = [1 if c == y else 0 for c in ar.depth_candidates[t]]
        omegas.append(omega)
        eads.append(analysis.ead(omega))
        stabs.append(analysis.ead_stable(omega))
    return omegas, eads, stabs


# -------------------------------------------------------------------------------------
# depth exploration over one sequence (section 3.2)
# -------------------------------------------------------------------------------------

@dataclass
class NodeRecord:
    """One lattice node's evaluation (for comparison with the GPU library)."""
    round: int
    q: int
    node: int
    stage: int
    plen: int
    target_pos: int
    token: int
    margin: float
    masked: List[int]
    logits: Optional[np.ndarray] = None


@dataclass
class CommitRecord:
    token: int
    kstar: int
    rounds: int          # rounds since the previous commit (k*(t-1) + 1 after the first)
    p_c: int             # commit position


@dataclass
class DEXResult:
    tokens: List[int]
    commits: List[CommitRecord]
    nodes: List[NodeRecord]
    rounds: int
    layer_passes: int    # sum over rounds of d_{deepest live stage}: layers one GPU streams
    node_layers: int     # sum over nodes of the layers of their stage (compute work)

    def depth_charges(self, X: Sequence[int]) -> List[int]:
        """d_{k*(t)} for every committed token: the depth-side charge (Eq. 12's W)."""
        return [X[c.kstar] for c in self.commits]


def dex_generate(model, prompt: Sequence[int], X: Sequence[int], T: int, rule: Rule = Rule(),
                 use_decs: bool = True, seq: int = 0, keep_logits: bool = False,
                 max_branch: int = 0, adapters: Optional[Sequence[Dict]] = None, cache=None) -> DEXResult:
    """Depth exploration decoding of T tokens for one sequence (section 3.2), with a trace.

    The decode is a series of exploration cycles, one per committed token.  A cycle is
    centred on the commit position p_c and runs explorer rounds until the anchor path
    reaches the final depth; the final-depth anchor token is committed, and the lattice
    is cut down to the part whose prefix is still valid (see ``_exploration_cycle``).

    max_branch > 0 builds a sparse lattice (the pruning of low-value branches that the
    paper's discussion of expansion growth proposes, with the final-depth commit kept): a
    node exists only if its parent does and its path holds at most max_branch position
    moves, i.e. it speculates at most that many tokens ahead of the commit.  The anchor
    chain has none and always exists, so the committed stream is unchanged.

    adapters: one inducing adapter per non-final depth X[0..N-2] (Appendix C.2; fp64 arrays
    as oracle.model.apply_adapter takes them) applied before the shared exit head of the
    nodes at those stages; the final depth keeps the plain exit, so commits are unchanged.

    cache: a ``prefill`` of the same prompt with room for P + T + N + 1 positions, or None to
    prefill here.
    """
    N = len(X)
    assert X[-1] == model.L and list(X) == sorted(set(X))
    committed = [int(t) for t in prompt]
    # the committed context: every prompt position but the last has its KV state; the last
    # prompt token is the input of the first anchor (the root of the first lattice)
    if cache is None:
        cache = prefill(model, committed, len(committed) + T + N + 1)
    res = DEXResult([], [], [], 0, 0, 0)
    lattice: Dict[int, int] = {}      # explore buffer: heap index -> candidate token
    rounds_done = 0                   # explorer rounds completed since the last commit
    while len(res.tokens) < T:
        y, kstar, lattice, rounds_done = _exploration_cycle(
            model, committed, cache, X, lattice, rounds_done, rule, use_decs, seq, keep_logits, max_branch,
            adapters, res)
        res.tokens.append(y)
        committed.append(y)
    return res


def _exploration_cycle(model, committed: List[int], cache, X: Sequence[int], lattice: Dict[int, int],
                       rounds_done: int, rule: Rule, use_decs: bool, seq: int, keep_logits: bool,
                       max_branch: int, adapters, res: DEXResult):
    """One cycle around the commit position p_c = len(committed) (section 3.2).

    Rounds continue from ``rounds_done`` (what survived the previous collapse).  In the
    round after r completed rounds, every existing node of level r of the binary lattice
    is evaluated: a node continues its slot chain one explorer deeper (a depth child) or
    opens a new slot at the next position with its parent's candidate as prefix (a
    position child).  Its hidden state is the model run on its prefix -- the committed
    tokens plus the candidates of the position moves on its path -- to the boundary d_s of
    its explorer s; its candidate comes from the shared exit head under depth-coupled
    sampling.  After N rounds the anchor path (the slot chain of p_c itself) has reached
    the final depth: its final-depth token is committed, the shallowest anchor depth that
    already proposed it is the accepted branch k*, and the lattice collapses onto it.

    Returns (committed token, k*, collapsed lattice, rounds it has already completed).
    """
    N = len(X)
    p_c = len(committed)
    # the anchor path at every depth: the committed prefix through the model, as AR computes it
    anchor_states = model.forward([committed[-1]], p_c - 1, cache, keep_depths=True)
    rounds_in_cycle = 0
    while True:
        level_q = rounds_done
        evaluated: Dict[int, int] = {}
        for i in level_nodes(level_q):
            if i > 0 and parent(i) not in lattice:
                continue                  # its branch was discarded (or never materialised)
            prefix = [lattice[a] for a in branch_parents(i)]
            if max_branch > 0 and len(prefix) > max_branch:
                continue
            s = stage(i)
            if prefix:
                h = model.forward(prefix, p_c, cache, depth=X[s])[-1:]
            else:
                h = anchor_states[X[s] - 1]
            res.node_layers += X[s] - (X[s - 1] if s > 0 else 0)
            ad = adapters[s] if adapters is not None and s < N - 1 else None
            z = model.exit_logits(h, ad)[0]
            shallower = [lattice[a] for a in prior_nodes(i) if a in lattice]
            tok, mg, excluded = depth_coupled_token(z, shallower, s == N - 1, rule, seq, p_c + len(prefix),
                                                    enabled=use_decs)
            evaluated[i] = tok
            res.nodes.append(NodeRecord(res.rounds, level_q, i, s, len(prefix), p_c + len(prefix), tok, mg,
                                        excluded, z if keep_logits else None))
        lattice.update(evaluated)
        res.layer_passes += X[level_q]
        res.rounds += 1
        rounds_in_cycle += 1
        if level_q < N - 1:
            rounds_done += 1
            continue
        y, kstar = select_commit([lattice[anchor_node(k)] for k in range(N)])
        res.commits.append(CommitRecord(y, kstar, rounds_in_cycle, p_c))
        lattice, rounds_done = collapse(lattice, N, kstar)
        return y, kstar, lattice, rounds_done


def select_commit(anchor_tokens: Sequence[int]) -> Tuple[int, int]:
    """Section 3.2, commit: the final-depth anchor token u_{N-1} is committed; the accepted
    branch is the shallowest anchor depth k whose candidate u_k equals it (k = N-1 when
    no shallower depth did)."""
    y = int(anchor_tokens[-1])
    kstar = next(k for k, u in enumerate(anchor_tokens) if u == y)
    return y, kstar


def collapse(lattice: Dict[int, int], N: int, kstar: int) -> Tuple[Dict[int, int], int]:
    """Keep only the nodes whose prefix is the new committed prefix; return them
    re-indexed from the new root, and the rounds the new lattice has already completed.

    The valid nodes are the subtree of m = P(b_{k*}), the position child of the accepted
    branch: every other node's prefix holds a token that was not committed.  m was created
    k*+1 rounds into the cycle, so its subtree covers N - k* - 1 completed rounds.  With the
    fallback branch (k* = N-1) nothing survives, and neither when a sparse lattice never
    materialised m.
    """
    if kstar == N - 1:
        return {}, 0
    m = position_child(anchor_node(kstar))
    if m not in lattice:
        return {}, 0
    remap = subtree_remap(m, N - 1)
    kept = {new: lattice[old] for old, new in remap.items() if old in lattice}
    return kept, N - kstar - 1
