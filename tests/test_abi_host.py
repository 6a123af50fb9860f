"""CPU tests of the C ABI: the library loads, exports every declared symbol, rejects bad
arguments, and its host-side lattice scheduler reproduces the oracle's Algorithm 1."""
import os
import re

import pytest

import dex_inputs as di
from conftest import ROOT, tiny_model
from oracle import dex as odex

dexlib = pytest.importorskip("lossless_depth_adaptive_gb300")


def _lib():
    try:
        return dexlib.lib()
    except dexlib.DexLibraryMissing:
        from lossless_depth_adaptive_gb300 import build
        build.build()
        return dexlib.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "dex.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dex_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    L = _lib()
    syms = declared_symbols()
    assert len(syms) >= 20
    for s in syms:
        assert hasattr(L, s), s
        assert s in dexlib.SIGNATURES, f"{s} has no binding"


def test_strerror_and_bad_arguments():
    L = _lib()
    assert L.dex_strerror(0) == b"ok"
    assert b"capacity" in L.dex_strerror(-4)
    import ctypes as C
    h = C.c_void_p()
    assert L.dex_init(None, None, 0, None, None, C.byref(h)) == dexlib.DEX_EINVAL
    lat = C.c_void_p()
    assert L.dex_lattice_new(dexlib.i32([4, 2]), 2, 1, 1, 0, C.byref(lat)) == dexlib.DEX_EINVAL   # not increasing
    assert L.dex_lattice_new(dexlib.i32([4]), 1, 0, 1, 0, C.byref(lat)) == dexlib.DEX_EINVAL      # batch 0
    assert L.dex_lattice_new(dexlib.i32([4]), 1, 1, 1, -1, C.byref(lat)) == dexlib.DEX_EINVAL     # negative cap
    assert L.dex_exit_head_decs(None, 1, 128, None, 1e-5, None, 10, None, None, 0, 1.0, 0, None, None,
                                None) == dexlib.DEX_EINVAL


def _drive_lattice_with_oracle(X, alpha, tied, sample, use_decs, T=12, max_branch=0):
    _lib()
    _, _, m = tiny_model(alpha, tied)
    prompt = di.gen_prompts(di.TINY, 1, 32)[0].tolist()
    rule = odex.Rule(sample=sample, tau=0.7, seed=3)
    ref = odex.dex_generate(m, prompt, X, T, rule=rule, use_decs=use_decs, max_branch=max_branch)
    N = len(X)
    lat = dexlib.Lattice(X, 1, use_decs, max_branch)
    lat.start(0, len(prompt), prompt[-1])
    rounds = {}
    by_heap_prev = {}
    for nd in ref.nodes:
        rounds.setdefault(nd.round, []).append(nd)
    commits = iter(ref.commits)
    p_c = len(prompt)
    last = prompt[-1]
    for r in range(ref.rounds):
        plan = lat.plan()
        want = rounds[r]
        assert sorted(p["heap"] for p in plan) == sorted(n.node for n in want)
        by_heap = {n.node: n for n in want}
        slots = set()
        for p in plan:
            o = by_heap[p["heap"]]
            assert (p["stage"], p["plen"], p["target_pos"]) == (o.stage, o.plen, o.target_pos)
            assert p["pos"] == p_c - 1 + p["plen"] and p["c_end"] == p_c
            assert sorted(set(p["prior"])) == o.masked
            assert p["unmasked"] == (1 if p["stage"] == N - 1 else 0)
            assert p["n_tail"] == p["plen"]
            if p["plen"]:
                assert p["tail"][-1] == p["slot"]           # own position is the last tail entry
            assert p["kv_commit"] == (1 if odex.slot_root(p["heap"]) == 0 else 0)
            if p["heap"] == 0:
                assert p["token"] == last                    # root input: last committed token
            elif p["stage"] == 0:
                assert p["token"] == by_heap_prev[odex.parent(p["heap"])]   # parent's candidate
            else:
                assert p["token"] == -1
            slots.add((odex.slot_root(p["heap"]), p["slot"]))
        # one pool slot per slot chain, distinct across chains
        assert len({s for _, s in slots}) == len({r for r, _ in slots})
        stages = [p["stage"] for p in plan]
        assert stages == sorted(stages)                      # grouped by stage
        committed, kstar, jobs = lat.update([by_heap[p["heap"]].token for p in plan])
        by_heap_prev.update({h: n.token for h, n in by_heap.items()})
        if committed[0] >= 0:
            c = next(commits)
            last = c.token
            assert (committed[0], kstar[0]) == (c.token, c.kstar)
            m_root = odex.position_child(odex.anchor_node(c.kstar)) if c.kstar < N - 1 else None
            if m_root is not None and m_root in by_heap_prev:   # survivors re-indexed: i -> i - m 2^h
                remap = odex.subtree_remap(m_root, N - 1)
                by_heap_prev = {remap[o]: t for o, t in by_heap_prev.items() if o in remap}
                assert jobs == [(0, jobs[0][1], p_c, X[N - c.kstar - 2])]
            else:   # fallback, or a sparse lattice that never materialised m: nothing survives
                by_heap_prev = {}
                assert jobs == []
            p_c += 1
        q, pc, used = lat.state(0)
        assert pc == p_c and used <= 2 ** (N - 1)
    assert next(commits, None) is None


@pytest.mark.parametrize("X", [[2, 4, 6, 8], [4, 8], [1, 2, 3, 4, 5, 6, 7, 8], [8]])
@pytest.mark.parametrize("alpha,tied", [(0.3, False), (1.0, False)])
def test_lattice_scheduler_matches_oracle(X, alpha, tied):
    _drive_lattice_with_oracle(X, alpha, tied, sample=False, use_decs=True)


@pytest.mark.parametrize("X", [[2, 4, 6, 8], [1, 2, 3, 4, 5, 6, 7, 8]])
@pytest.mark.parametrize("cap", [1, 2])
def test_sparse_lattice_scheduler_matches_oracle(X, cap):
    """The speculation-capped lattice plans exactly the oracle's nodes, commits and collapses."""
    _drive_lattice_with_oracle(X, 1.0, False, sample=False, use_decs=True, max_branch=cap)
    _drive_lattice_with_oracle(X, 0.3, False, sample=True, use_decs=True, max_branch=cap)


def test_lattice_scheduler_sampled_and_vanilla():
    _drive_lattice_with_oracle([2, 4, 6, 8], 1.0, False, sample=True, use_decs=True)
    _drive_lattice_with_oracle([2, 4, 6, 8], 1.0, False, sample=False, use_decs=False)


def test_lattice_batch_of_sequences_is_independent():
    _lib()
    X = [2, 4, 6, 8]
    lat = dexlib.Lattice(X, 3, True)
    for b in range(3):
        lat.start(b, 10 + b, 7 + b)
    plan = lat.plan()
    assert [p["seq"] for p in plan] == [0, 1, 2]
    committed, _, _ = lat.update([1, 2, 3])
    assert committed == [-1, -1, -1]
    plan = lat.plan()
    # level 1: stage-0 nodes of every sequence first, then stage-1 nodes
    assert [(p["stage"], p["seq"], p["heap"]) for p in plan] == [(0, 0, 2), (0, 1, 2), (0, 2, 2),
                                                                 (1, 0, 1), (1, 1, 1), (1, 2, 1)]
    # the position child of the root takes the root's candidate as input token
    assert [p["token"] for p in plan if p["stage"] == 0] == [1, 2, 3]


def test_error_codes_match_the_header():
    """The binding's DEX_* constants equal include/dex.h's enum, and every code has its own
    message from dex_strerror."""
    src = open(os.path.join(ROOT, "include", "dex.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    codes = {name: int(val) for name, val in re.findall(r"\b(DEX_[A-Z]+)\s*=\s*(-?\d+)", src)}
    assert {"DEX_OK", "DEX_EINVAL", "DEX_ENOMEM", "DEX_ECUDA", "DEX_ECAPACITY", "DEX_ETIMEOUT", "DEX_ESTATE",
            "DEX_ENODEV", "DEX_ERANGE"} <= set(codes)
    for name, val in codes.items():
        assert getattr(dexlib, name) == val, name
    L = _lib()
    msgs = {L.dex_strerror(v) for v in codes.values()}
    assert len(msgs) == len(codes) and b"unknown error" not in msgs
    assert L.dex_strerror(-99) == b"unknown error"
