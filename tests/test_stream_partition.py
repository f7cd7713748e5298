"""Host check of the stream-K work split used by the decode GEMV: CTA g of G
takes units [g U / G, (g + 1) U / G); with the grid cut to min(G, U) every CTA
owns a unit, each (segment, tile) job gets exactly one epilogue (by its only
holder, or by the last of its holders through the split-tile counter), and the
partial slots read by that last holder are the ones its co-holders wrote.  The
rule is restated here from the kernel's description, in plain Python."""
import random


def _rb(g, G, U):
    return g * U // G


def _cta_of(u, G, U):
    return ((u + 1) * G - 1) // U


def _simulate(grid, U, ks):
    G = min(grid, U)
    epilogues, slots, counters = {}, {}, {}
    for g in range(G):
        u0, u1 = _rb(g, G, U), _rb(g + 1, G, U)
        assert u1 > u0
        i = 0
        while i < u1 - u0:
            job = (u0 + i) // ks
            jb, je = job * ks, job * ks + ks
            if jb >= u0 and je <= u1:
                epilogues[job] = epilogues.get(job, 0) + 1
            else:
                which = 0 if jb <= u0 else 1
                assert (g, which) not in slots
                slots[(g, which)] = job
                ga, gb = _cta_of(jb, G, U), _cta_of(je - 1, G, U)
                counters[job] = counters.get(job, 0) + 1
                if counters[job] - 1 == gb - ga:
                    for c in range(ga, gb + 1):
                        assert slots[(c, 0 if jb <= _rb(c, G, U) else 1)] == job
                    epilogues[job] = epilogues.get(job, 0) + 1
            i = min(je, u1) - u0
    return epilogues


def test_every_unit_has_one_owner():
    for G in list(range(1, 70)) + [456, 576]:
        for U in list(range(1, 130)) + [3072, 22528]:
            for u in (range(U) if U < 200 else (0, U // 3, U - 1)):
                g = _cta_of(u, min(G, U), U)
                assert _rb(g, min(G, U), U) <= u < _rb(g + 1, min(G, U), U)


def test_every_job_gets_exactly_one_epilogue():
    rng = random.Random(5)
    cases = [(64, 52, 2), (456, 3072, 16), (304, 22528, 16), (456, 1536, 8), (576, 24, 1)]
    cases += [(rng.randint(1, 600), 0, rng.choice([1, 2, 3, 8, 16, 32, 64])) for _ in range(400)]
    for G, U, ks in cases:
        if U == 0:
            U = rng.randint(1, 300) * ks
        ep = _simulate(G, U, ks)
        assert all(ep.get(j, 0) == 1 for j in range(U // ks)), (G, U, ks)
