"""The scoreboard a stage boundary must have, rebuilt from the oracle's brute-force dependency
enumeration alone (test infrastructure; it shares nothing with the library's builder).

The pages initialise one counter per consumer tile from the dependency array (CTA-Pipelining,
section III-A).  The library shares one counter among consumer tiles that become ready together;
what each counter must wait for follows from the enumeration:
  - the partition: with raster_group <= 1, classes of consumer tiles whose enumerated producer sets
    are equal (numbered by smallest member, members ascending); with g > 1, the consumer tiles of g
    consecutive row panels, listed column by column;
  - a group's target: the size of the union of its members' producer sets, times the releases one
    producer tile makes per run (split-K slices x epilogue warps);
  - per producer tile: the groups of the consumer tiles it feeds, ascending.
"""
import numpy as np


def expected(oracle, M, n_out, n_next, bm, bn_p, bn_c, raster_group, releases):
    off, tgt, _ = oracle.deps(M, n_out, n_next, bm, bn_p, bm, bn_c)
    P = len(off) - 1
    tiles_n = -(-n_next // bn_c)
    C = -(-M // bm) * tiles_n
    prods = [set() for _ in range(C)]
    for p in range(P):
        for c in tgt[off[p]:off[p + 1]]:
            prods[int(c)].add(p)
    groups = []
    if raster_group <= 1:
        first = {}
        for c in range(C):
            key = tuple(sorted(prods[c]))
            if key not in first:
                first[key] = len(groups)
                groups.append([])
            groups[first[key]].append(c)
    else:
        panels = -(-C // tiles_n)
        for m0 in range(0, panels, raster_group):
            groups.append([m * tiles_n + n for n in range(tiles_n)
                           for m in range(m0, min(panels, m0 + raster_group)) if m * tiles_n + n < C])
    cons_grp = np.zeros(C, np.int32)
    for g, mem in enumerate(groups):
        cons_grp[mem] = g
    grp_off = np.cumsum([0] + [len(m) for m in groups]).astype(np.int32)
    grp_mem = np.array([c for m in groups for c in m], np.int32)
    grp_target = np.array([len(set().union(*(prods[c] for c in m))) * releases for m in groups], np.int32)
    pg = [sorted({int(cons_grp[int(c)]) for c in tgt[off[p]:off[p + 1]]}) for p in range(P)]
    pg_off = np.cumsum([0] + [len(x) for x in pg]).astype(np.int32)
    pg_tgt = np.array([g for x in pg for g in x], np.int32)
    return {"producers": P, "consumers": C, "groups": len(groups), "releases_per_producer": releases,
            "pg_off": pg_off, "pg_tgt": pg_tgt, "grp_off": grp_off, "grp_mem": grp_mem,
            "grp_target": grp_target, "cons_grp": cons_grp}


def assert_equal(got, want):
    for k, v in want.items():
        if isinstance(v, np.ndarray):
            assert np.array_equal(np.asarray(got[k]), v), k
        else:
            assert got[k] == v, k
