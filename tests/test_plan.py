"""The bf16 decode work split (host arithmetic shared with the kernel).

The batch's pages are laid end to end and cut into equal ranges, one per
2-CTA cluster; these tests check, without a GPU, the properties the kernel
and its combine step rely on: every page of every unit is processed exactly
once, no piece is empty, partial slots are unique and in range, and a unit's
pieces sit in consecutive clusters g_first..g_last (so the combine finds
exactly the slots that were written).
"""

import math
import random

import pytest

from mla_latent_kv_71_b300 import mla, workloads


def unit_pages(lens, T, H, causal):
    # units lie on the line in the order u = (t * HG + hg) * B + b
    HG = (H + 127) // 128
    pages = []
    for t in range(T):
        for hg in range(HG):
            for n in lens:
                v = max(0, n - (T - 1 - t)) if causal else n
                pages.append(math.ceil(v / 64))
    return pages


def launched_clusters(pages, clusters):
    """One cluster per unit when all non-empty units have the same pages n,
    there are at most `clusters` of them, and n exceeds the largest range of
    the cut over all clusters by at most 16 pages; else `clusters`."""
    ne = [n for n in pages if n]
    if not ne or len(set(ne)) != 1 or len(ne) > clusters:
        return clusters
    total = sum(ne)
    C = 3 if total >= 8 * clusters else 0
    V = total + C * (len(ne) - 1)
    return len(ne) if ne[0] - math.ceil(V / clusters) <= 16 else clusters


def check_plan(lens, T, H, max_pages, causal, clusters):
    pieces = mla.decode_plan(lens, T, H, max_pages, causal, clusters)
    HG = (H + 127) // 128
    U = len(lens) * T * HG
    pages = unit_pages(lens, T, H, causal)
    clusters = launched_clusters(pages, clusters)
    total = sum(pages)
    G = min(clusters, total)
    seen = {}
    slots = set()
    by_unit = {}
    for p in pieces:
        assert 0 <= p["cluster"] < G
        assert p["lp1"] > p["lp0"], p
        for lp in range(p["lp0"], p["lp1"]):
            key = (p["unit"], lp)
            assert key not in seen, key
            seen[key] = p["cluster"]
        whole = p["g_first"] == p["g_last"]
        assert (p["slot"] == -1) == whole
        if not whole:
            assert p["slot"] == p["cluster"] + p["unit"]
            assert p["slot"] not in slots
            assert 0 <= p["slot"] < G + U
            slots.add(p["slot"])
        by_unit.setdefault(p["unit"], []).append(p)
    for u, n in enumerate(pages):
        for lp in range(n):
            assert (u, lp) in seen, (u, lp)
        if n:
            cl = sorted(p["cluster"] for p in by_unit[u])
            assert cl == list(range(by_unit[u][0]["g_first"], by_unit[u][0]["g_last"] + 1))
    # Ranges are equal cuts of the virtual line, on which each non-empty unit
    # after the first is preceded by C virtual pages (C = 3 on lines of at
    # least 8 pages per cluster, else 0): no cluster holds more than
    # ceil(V / G) real pages, every cluster holds some, and clusters whose
    # range holds a unit boundary hold fewer real pages on average than those
    # without (a range that starts or ends inside a gap holds fewer too).
    nonempty = sum(1 for n in pages if n)
    C = 3 if total >= 8 * clusters else 0
    V = total + C * (nonempty - 1) if nonempty else 0
    per = {}
    for p in pieces:
        per[p["cluster"]] = per.get(p["cluster"], 0) + p["lp1"] - p["lp0"]
    if total:
        assert max(per.values()) <= math.ceil(V / G)
        assert len(per) == G
        if C:
            npieces = {}
            for p in pieces:
                npieces[p["cluster"]] = npieces.get(p["cluster"], 0) + 1
            one = [per[g] for g in per if npieces[g] == 1]
            more = [per[g] for g in per if npieces[g] > 1]
            if one and more:
                assert sum(more) / len(more) < sum(one) / len(one)
    return pieces


@pytest.mark.parametrize("lens,T,H", [
    ([1, 65, 200], 1, 128), ([64, 128, 640, 1000], 1, 128), ([2, 129], 2, 128),
    ([33, 64, 300], 1, 16), ([70, 130], 1, 200), ([3, 250], 3, 128), ([0, 70, 5], 1, 128),
    ([1], 1, 128), ([0, 0], 1, 128),
])
@pytest.mark.parametrize("clusters", [1, 3, 74, 500])
def test_small_plans(lens, T, H, clusters):
    check_plan(lens, T, H, max(1, math.ceil(max(lens) / 64)), T > 1, clusters)


@pytest.mark.parametrize("name", ["decode_b64_h128_l4096", "ragged_b128_l16k", "long_b4_l128k",
                                  "mtp_b32_t2_l8192", "smallhead_b64_h16_l32k"])
def test_workload_plans(name):
    spec = workloads.WORKLOADS[name]
    lens = workloads.workload_lens(spec)
    check_plan(lens, spec["T"], spec["H"], math.ceil(max(lens) / 64), spec["T"] > 1, 74)


def test_random_plans():
    rng = random.Random(0)
    for _ in range(200):
        B = rng.randint(1, 40)
        lens = [rng.choice([0, 1, 63, 64, 65, rng.randint(0, 5000)]) for _ in range(B)]
        T = rng.randint(1, 3)
        H = rng.choice([16, 128, 129, 300])
        mp = max(1, math.ceil(max(lens) / 64))
        check_plan(lens, T, H, mp, rng.random() < 0.5, rng.choice([1, 2, 7, 74, 148]))


def test_uniform_batch_is_not_split_when_clusters_divide_it():
    pieces = check_plan([4096] * 64, 1, 128, 64, False, 64)
    assert all(p["slot"] == -1 for p in pieces)


def test_uniform_headline_batch_takes_one_cluster_per_sequence():
    """64 sequences of 4096 on 74 clusters: 64 clusters, no unit cut (the
    step without the merge kernel measured faster); 64 x 32768 with 16
    heads keeps all 74 clusters and cuts units (512 pages per cluster would
    be 69 more than the cut's largest range)."""
    pieces = check_plan([4096] * 64, 1, 128, 64, False, 74)
    assert len({p["cluster"] for p in pieces}) == 64
    assert all(p["slot"] == -1 for p in pieces)
    pieces = check_plan([32768] * 64, 1, 16, 512, False, 74)
    assert len({p["cluster"] for p in pieces}) == 74
    assert any(p["slot"] != -1 for p in pieces)
