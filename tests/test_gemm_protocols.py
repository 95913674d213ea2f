"""Randomised interleaving checks of the tcgen05 matmul kernels' hand-offs
(CPU only; no GPU code runs): the CTA-pair matmul (gemm_tc_pair_kernel),
its split-K reduction in split order across CTA pairs, and the few-row
matmul's cluster reduction through distributed shared memory
(gemm_rows_tc_kernel), as written in csrc/k_gemm_tc.cu.

The simulator (protocol_sim.py) checks each interleaving for deadlock,
aliased phase waits, arrivals landing in another phase, races on shared
memory, tensor memory and staging buffers, and work in flight at exit.
Planted mistakes in the models show that the checks fire.
"""
import pytest

from protocol_sim import Sim, find

EPI_WARPS = 8          # epilogue warps per CTA
PAIR_STAGES = {False: 6, True: 5}   # operand ring depth without / with the aux staging


# -------------------------------------------------------------- CTA pair
def gemm_pair(ntiles, seed, plant=None, aux=False, gelu2=False, ew=EPI_WARPS, nch=2, ctas=2):
    """One cluster of two CTAs running ntiles output tiles (256 x 256) in
    turn.  Per CTA a producer thread loads its half of the A and B k-tiles
    into ring stage it % S once the leader's MMAs have released the stage
    (the release is committed to both CTAs' empty barriers); both halves'
    bytes complete the leader's full barrier, whose one arrival is the
    leader's expect-tx.  The leader's MMA thread waits for a free
    accumulator (two in TMEM), runs the tile's k-tiles from both CTAs'
    stages into both CTAs' tensor memory, and commits the stage releases
    and the accumulator to both CTAs.  Each CTA's epilogue warps wait for
    their CTA's accumulator, read it chunk by chunk through a staging
    buffer (TMA stores from it; a buffer is rewritten only after the warp's
    earlier stores have read it), and arrive on the leader's accumulator
    barrier.  With aux, each chunk's auxiliary tile is loaded into one of
    two staging buffers one chunk ahead and overwritten in place by the
    result.  At the end the producers wait for every release still to come,
    the MMA thread for every accumulator release, the warps for their
    stores.  With ctas=1 the same protocol runs in one CTA (gemm_tc_kernel,
    the 128-row tiles of narrow outputs)."""
    sim = Sim(seed, plant)
    R = range(ctas)
    S = PAIR_STAGES[aux]
    nkt = [sim.rnd.randint(1, 2 * S) for _ in range(ntiles)]
    for s in range(S):
        sim.bar("full%d" % s, 1 + ctas)  # leader's arrive.expect_tx + the bytes of each CTA
        for r in R:
            sim.bar("empty%d_%d" % (r, s))
    for a in (0, 1):
        sim.bar("accempty%d" % a, ctas * ew)
        for r in R:
            sim.bar("accfull%d_%d" % (r, a))
    for r in R:
        for w in range(ew):
            for b in (0, 1):
                sim.bar("aux%d_%d_%d" % (r, w, b))

    def producer(r):
        it = 0
        for t in range(ntiles):
            for _ in range(nkt[t]):
                s, k = it % S, it // S
                if not (plant == "peer_unguarded" and r == 1):
                    yield from sim.wait("empty%d_%d" % (r, s), k - 1)
                if r == 0:
                    sim.arrive("full%d" % s, phase=k)
                sim.tma("full%d" % s, "A%d_%d" % (r, s), "B%d_%d" % (r, s), phase=k)
                it += 1
        if plant != "no_release_drain":
            for d in range(max(0, it - S), it):
                yield from sim.wait("empty%d_%d" % (r, d % S), d // S)

    def issuer():
        it = 0
        for ti in range(ntiles):
            a = ti & 1
            if plant != "acc_unguarded":
                yield from sim.wait("accempty%d" % a, (ti >> 1) - 1)
            for _ in range(nkt[ti]):
                s, k = it % S, it // S
                yield from sim.wait("full%d" % s, k)
                sim.mma(reads=[x % (r, s) for r in R for x in ("A%d_%d", "B%d_%d")],
                        writes=["acc%d_%d" % (r, a) for r in R])
                for r in R:
                    sim.commit("empty%d_%d" % (r, s), phase=k)
                it += 1
            for r in R:
                sim.commit("accfull%d_%d" % (r, a), phase=ti >> 1)
        for d in range(max(0, ntiles - 2), ntiles):
            yield from sim.wait("accempty%d" % (d & 1), d >> 1)

    def epilogue(r, w):
        me = (r, w)
        loads = [0, 0]   # loads into each aux staging buffer so far

        def aux_load(b):
            sim.tma("aux%d_%d_%d" % (r, w, b), "stg%d_%d_%d" % (r, w, b), phase=loads[b])
            loads[b] += 1

        for ti in range(ntiles):
            a = ti & 1
            acc = "acc%d_%d" % (r, a)
            if aux:
                yield from sim.wait_read(me)
                aux_load(0)
                yield from sim.wait("accfull%d_%d" % (r, a), ti >> 1)
                t_acc = sim.t
                for c in range(nch):
                    b = c & 1
                    if c + 1 < nch:
                        if plant != "aux_reload_unguarded":
                            yield from sim.wait_read(me)
                        aux_load((c + 1) & 1)
                    yield from sim.work(1, 3)                       # tcgen05.ld of the chunk
                    yield from sim.wait("aux%d_%d_%d" % (r, w, b), loads[b] - 1)
                    t0 = sim.t
                    yield from sim.work(1, 3)
                    sim.touch("warp", "w", t0, "stg%d_%d_%d" % (r, w, b))
                    sim.store(me, "stg%d_%d_%d" % (r, w, b))
                    t1 = sim.t
                    yield from sim.work(0, 2)                       # column sums read the staging rows
                    sim.touch("warp", "r", t1, "stg%d_%d_%d" % (r, w, b))
            else:
                yield from sim.wait("accfull%d_%d" % (r, a), ti >> 1)
                t_acc = sim.t
                for c in range(nch):
                    if plant != "staging_unguarded":
                        yield from sim.wait_read(me)
                    yield from sim.work(1, 3)                       # tcgen05.ld of the chunk
                    t0 = sim.t
                    yield from sim.work(1, 3)
                    bufs = ["stg%d_%d_0" % (r, w)] + (["stg%d_%d_1" % (r, w)] if gelu2 else [])
                    sim.touch("warp", "w", t0, *bufs)
                    for b in bufs:                                  # one bulk group per output
                        sim.store(me, b)
            sim.touch("warp", "r", t_acc, acc)
            sim.arrive("accempty%d" % a, phase=ti >> 1)
        if plant != "no_store_drain":
            yield from sim.wait_stores(me)

    actors = [producer(r) for r in R] + [issuer()]
    actors += [epilogue(r, w) for r in R for w in range(ew)]
    sim.run(actors)
    return sim.errors


TILES = [1, 2, 3, 4, 7]


@pytest.mark.parametrize("variant", [dict(), dict(aux=True), dict(gelu2=True), dict(aux=True, nch=4),
                                     dict(ctas=1), dict(ctas=1, nch=4)])
def test_pair_matmul_protocol(variant):
    for n in TILES:
        for seed in range(6):
            errs = gemm_pair(n, seed, ew=4, **variant)
            assert not errs, (variant, n, seed, errs[:3])


def test_pair_matmul_protocol_with_eight_epilogue_warps():
    for n in (1, 3):
        for seed in range(3):
            errs = gemm_pair(n, seed, aux=True)
            assert not errs, (n, seed, errs[:3])


@pytest.mark.parametrize("plant,kind,variant", [
    ("peer_unguarded", "race on A1_", {}),
    ("acc_unguarded", "race on acc", {}),
    ("staging_unguarded", "race on stg", {}),
    ("aux_reload_unguarded", "race on stg", dict(aux=True, nch=4)),
    ("no_store_drain", "in flight at exit", {}),
])
def test_pair_matmul_checker_finds_a_planted_mistake(plant, kind, variant):
    errs = find(gemm_pair, plant, kind, [2, 3, 5], seeds=8, ew=2, **variant)
    assert errs, plant


# -------------------------------------------------------------- split-K order
def splitk_order(npairs, seed, plant=None, regions=3, splits=3, capacity=None):
    """Split-K of the pair matmul reduced inside the kernel: tile t is split
    t // regions of output region t % regions; pair p runs tiles p, p +
    npairs, ... in turn.  A tile's epilogue waits until its region's flag
    (ld.acquire) equals its split, adds its part into the output, waits for
    its stores and hands the region on (st.release of split + 1, or 0 after
    the last split, so the flags are ready for the next launch).  The pairs
    become resident in any order, and the number that may be resident grows
    from a random start (the previous kernel still draining) to capacity;
    the host launches at most as many pairs as can be resident at once."""
    sim = Sim(seed, plant)
    cap_max = capacity if capacity is not None else npairs
    flags = [0] * regions
    order = {r: [] for r in range(regions)}
    total = splits * regions
    state = {"cap": sim.rnd.randint(1, cap_max), "resident": set(), "queue": list(range(npairs))}
    sim.rnd.shuffle(state["queue"])

    def scheduler():
        while state["queue"]:
            if state["cap"] < cap_max and sim.rnd.random() < 0.1:
                state["cap"] += 1
            while state["queue"] and len(state["resident"]) < state["cap"]:
                state["resident"].add(state["queue"].pop(0))
            yield

    def pair(p):
        while p not in state["resident"]:
            yield
        for t in range(p, total, npairs):
            split, region = t // regions, t % regions
            yield from sim.work(1, 6)                       # the tile's main loop
            while flags[region] != split:                   # flag_wait
                yield
            order[region].append(split)
            yield from sim.work(1, 4)                       # reduce-add, then wait for the stores
            last = split == splits - 1
            flags[region] = 0 if last and plant != "flag_not_reset" else split + 1
        state["resident"].discard(p)

    sim.run([scheduler()] + [pair(p) for p in range(npairs)], limit=20000)
    if not any("deadlock" in e for e in sim.errors):
        if any(flags):
            sim.errors.append("flag left set after the launch: %s" % flags)
        for r in range(regions):
            if order[r] != list(range(splits)):
                sim.errors.append("region %d reduced in order %s" % (r, order[r]))
    return sim.errors


def test_splitk_reduction_runs_in_split_order_and_resets_its_flags():
    for npairs in (1, 2, 3, 5, 9):
        for regions, splits in ((1, 4), (3, 2), (4, 4), (7, 3)):
            for seed in range(4):
                errs = splitk_order(npairs, seed, regions=regions, splits=splits)
                assert not errs, (npairs, regions, splits, seed, errs[:3])


def test_splitk_checker_finds_a_planted_mistake():
    assert find(splitk_order, "flag_not_reset", "flag left set", [2, 3])
    # more pairs than can be resident at once: a resident pair may wait
    # for a split that a pair still waiting for an SM owns
    errs = []
    for seed in range(20):
        errs += splitk_order(4, seed, regions=1, splits=4, capacity=2)
    assert any("deadlock" in e for e in errs)


# -------------------------------------------------------------- few-row matmul
def rows_cluster(ktiles, seed, plant=None, csize=4, stages=6):
    """gemm_rows_tc_kernel: a cluster of csize CTAs splits K; CTA r runs
    k-tiles [r * kps, min(ktiles, (r + 1) * kps)) (possibly none) through a
    stages-deep TMA -> MMA ring into tensor memory and commits 'done' after
    its last MMA (at once if it has none).  Its four warps wait for 'done',
    read the accumulator and, with csize > 1, write the partial sums to
    shared memory; after a cluster barrier the first CTA reads every other
    CTA's partial sums through distributed shared memory, and a second
    cluster barrier keeps the others resident until it has.  Every CTA then
    frees its tensor memory and exits."""
    sim = Sim(seed, plant)
    kps = -(-ktiles // csize)
    nks = [max(0, min(ktiles, r * kps + kps) - r * kps) for r in range(csize)]
    sim.bar("cs1", 4 * csize)
    sim.bar("cs2", 4 * csize)
    for r in range(csize):
        sim.bar("done%d" % r)
        sim.bar("end%d" % r, 4)
        for s in range(stages):
            sim.bar("full%d_%d" % (r, s))
            sim.bar("empty%d_%d" % (r, s))

    def producer(r):
        for i in range(nks[r]):
            s, k = i % stages, i // stages
            if i >= stages:
                yield from sim.wait("empty%d_%d" % (r, s), k - 1)
            sim.tma("full%d_%d" % (r, s), "W%d_%d" % (r, s), "X%d_%d" % (r, s), phase=k)

    def issuer(r):
        for i in range(nks[r]):
            s, k = i % stages, i // stages
            yield from sim.wait("full%d_%d" % (r, s), k)
            sim.mma(reads=("W%d_%d" % (r, s), "X%d_%d" % (r, s)), writes=("tm%d" % r,))
            sim.commit("empty%d_%d" % (r, s), phase=k)
        sim.commit("done%d" % r, phase=0)

    def warp(r, w):
        if w == 0:
            yield from producer(r)
        elif w == 1:
            yield from issuer(r)
        yield from sim.wait("done%d" % r, 0)
        t0 = sim.t
        yield from sim.work(1, 3)
        sim.touch("warp", "r", t0, "tm%d" % r)
        if csize > 1:
            t1 = sim.t
            yield from sim.work(1, 2)
            sim.touch("warp", "w", t1, "red%d" % r)
            if plant != "no_first_sync":
                sim.arrive("cs1", phase=0)
                yield from sim.wait("cs1", 0)
            if r == 0:
                t2 = sim.t
                yield from sim.work(1, 4)
                sim.touch("remote", "r", t2, *["red%d" % q for q in range(1, csize)])
            if plant != "no_second_sync":
                sim.arrive("cs2", phase=0)
                yield from sim.wait("cs2", 0)
        yield from sim.work(0, 2)                           # the first CTA writes the output
        sim.arrive("end%d" % r, phase=0)                    # __syncthreads, then exit
        yield from sim.wait("end%d" % r, 0)
        sim.touch("exit", "w", sim.t, "red%d" % r, "tm%d" % r, until=10 ** 9)   # freed

    sim.run([warp(r, w) for r in range(csize) for w in range(4)])
    return sim.errors


def test_few_row_matmul_cluster_reduction():
    for csize in (1, 2, 3, 8):
        for ktiles in (1, 2, 5, 12, 24):
            for seed in range(4):
                errs = rows_cluster(ktiles, seed, csize=csize)
                assert not errs, (csize, ktiles, seed, errs[:3])


@pytest.mark.parametrize("plant,kind", [("no_first_sync", "race on red"), ("no_second_sync", "race on red")])
def test_few_row_checker_finds_a_planted_mistake(plant, kind):
    assert find(rows_cluster, plant, kind, [4, 12], seeds=10)
