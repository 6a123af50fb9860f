"""Pins for the lattice indexing of oracle/dex.py: Figure 2 counts and brute-force paths.

Paths are strings over {D, P} (depth / position expansion) read from the root.
"""
import itertools
import pytest

from conftest import golden_lines
from oracle import dex


def heap_index(path):
    i = 0
    for c in path:
        i = 2 * i + (1 if c == "D" else 2)
    return i


def all_paths(max_len):
    for n in range(max_len + 1):
        for p in itertools.product("DP", repeat=n):
            yield "".join(p)


def test_figure2_counts():
    g = {}
    for ln in golden_lines("figure2_lattice_counts.txt"):
        g.setdefault(ln[0], []).extend(ln[1:])
    assert dex.depth_child(0) == int(g["depth_child_of_root"][0])
    assert dex.position_child(0) == int(g["position_child_of_root"][0])
    K = int(g["explorers"][0])
    # state q (q rounds done) materializes the first 2^q - 1 tokens
    state, size = int(g["state"][0]), int(g["state"][2])
    materialized = [i for q in range(state) for i in dex.level_nodes(q)]
    assert materialized == list(range(size)) and state == K
    assert sum(len(dex.level_nodes(q)) for q in range(4)) == int(g["cycle_max"][1])
    assert sum(len(dex.level_nodes(q)) for q in range(8)) == int(g["cycle_max"][3])
    assert len(dex.level_nodes(7)) == int(g["largest_round_batch"][1])


def test_indexing_against_path_strings():
    for path in all_paths(7):
        i = heap_index(path)
        assert dex.level(i) == len(path)
        trailing_d = len(path) - len(path.rstrip("D"))
        assert dex.stage(i) == trailing_d
        root_path = path.rstrip("D")
        assert dex.slot_root(i) == heap_index(root_path)
        # Prior(i): shallower members of the slot chain, nearest first
        assert dex.prior_nodes(i) == [heap_index(path[:len(path) - k]) for k in range(1, trailing_d + 1)]
        # branch parents: nodes immediately before each P move
        assert dex.branch_parents(i) == [heap_index(path[:j]) for j, c in enumerate(path) if c == "P"]
        if path:
            assert dex.parent(i) == heap_index(path[:-1])


@pytest.mark.parametrize("q", range(8))
def test_round_stage_counts(q):
    """Level q holds 2^(q-s-1) nodes at stage s < q (paths ending in P then s D moves)
    and the single anchor node at stage q."""
    stages = [dex.stage(i) for i in dex.level_nodes(q)]
    brute = [sum(1 for p in all_paths(q) if len(p) == q and len(p) - len(p.rstrip("D")) == s)
             for s in range(q + 1)]
    for s in range(q + 1):
        assert stages.count(s) == brute[s] == (2 ** (q - s - 1) if s < q else 1)
    # only the anchor reaches stage q at level q
    assert [i for i in dex.level_nodes(q) if dex.stage(i) == q] == [dex.anchor_node(q)]


def test_collapse_remap_closed_form():
    N = 6
    for k in range(N - 1):
        m = dex.position_child(dex.anchor_node(k))
        remap = dex.subtree_remap(m, N - 1)
        mpath = [p for p in all_paths(N - 1) if heap_index(p) == m][0]
        want = {}
        for p in all_paths(N - 1):
            if p.startswith(mpath):
                want[heap_index(p)] = heap_index(p[len(mpath):])
        assert remap == want
        # survivors keep their relative structure: stage and plen relative to m
        for old, new in remap.items():
            assert dex.stage(old) == dex.stage(new) or dex.slot_root(old) == m
            assert dex.level(new) <= N - 1 - dex.level(m)


def test_collapse_state_and_commit():
    N = 4
    B = {i: 100 + i for i in range(2 ** N - 1)}
    # y = u_3; make u_1 match -> k* = 1 -> survivors = subtree of 2^(k*+1) = 4
    B[dex.anchor_node(3)] = 7
    B[dex.anchor_node(1)] = 7
    B[dex.anchor_node(2)] = 7
    y, k = dex.select_commit([B[dex.anchor_node(j)] for j in range(N)])
    assert (y, k) == (7, 1)
    newB, q = dex.collapse(B, N, k)
    assert q == N - k - 1 == 2
    assert newB == {0: B[4], 1: B[9], 2: B[10]}
    # fallback
    B[dex.anchor_node(1)] = 8
    B[dex.anchor_node(2)] = 9
    y, k = dex.select_commit([B[dex.anchor_node(j)] for j in range(N)])
    assert (y, k) == (7, 3)
    assert dex.collapse(B, N, k) == ({}, 0)
