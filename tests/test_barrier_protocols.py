"""Randomised interleaving checks of the mbarrier protocols of the three
tensor-core attention kernels and of the LayerNorm backward's row ring
(CPU only; no GPU code runs).

Each kernel's roles are actors of the simulator in protocol_sim.py, which
checks every interleaving tried for deadlock, aliased phase waits,
arrivals that land in another phase, races on shared-memory and TMEM
buffers, and work still in flight at exit.  Warps that run the same code
are separate actors, so one may run a sub-block ahead of another.
Planted mistakes in the models show that the checks fire.  The models
follow attn_fwd_tc_kernel, attn_bwd_dkv_tc_kernel, attn_bwd_dq_tc_kernel
(csrc/k_attn_tc.cu) and layernorm_bwd_kernel (csrc/k_misc.cu); a change
to a kernel's hand-offs changes its model.
"""
import pytest

from protocol_sim import Sim, find

# warps and ring stages as the kernels are compiled: 8 softmax warps and 3
# key/value stages (forward); 16 compute warps and 4 query stages (dK/dV);
# 8 compute warps, 3 key and 2 value stages (dQ)
FWD_WARPS, FWD_STAGES = 8, 3
DKV_WARPS, DKV_STAGES = 16, 4
DQ_WARPS, DQ_K_STAGES, DQ_V_STAGES = 8, 3, 2


# -------------------------------------------------------------- forward
def forward(nsub, seed, plant=None, nsoft=FWD_WARPS, stages=FWD_STAGES):
    """Loader warp: q once, then k(j), v(j) into ring stage j % stages once
    S(j - stages), PV(j - stages) have read it.  MMA warp: S(0), S(1), then
    per sub-block PV(j) once P(j) is written and S(j + 2) after it.  Softmax
    warps: S(j) -> P(j) in shared memory (after PV(j - 2) has read that
    buffer), with an occasional rescale of O in tensor memory once PV(j - 1)
    is done; O read at the end."""
    sim = Sim(seed, plant)
    sim.bar("q")
    for s in range(stages):
        for n in ("kf%d", "vf%d", "ke%d", "ve%d"):
            sim.bar(n % s)
    for i in range(2):
        sim.bar("s%d" % i)
        sim.bar("o%d" % i)
        sim.bar("p%d" % i, nsoft)
    if plant == "one_p_barrier":   # P(j) written: one barrier for both buffers
        P, Pk = (lambda j: "p0"), (lambda j: j)
    else:
        P, Pk = (lambda j: "p%d" % (j & 1)), (lambda j: j >> 1)

    def loader():
        sim.tma("q", "sQ", phase=0)
        for j in range(nsub):
            s = j % stages
            if j >= stages and plant != "k_refill_unguarded":
                yield from sim.wait("ke%d" % s, j // stages - 1)
            sim.tma("kf%d" % s, "sK%d" % s, phase=j // stages)
            if j >= stages:
                yield from sim.wait("ve%d" % s, j // stages - 1)
            sim.tma("vf%d" % s, "sV%d" % s, phase=j // stages)

    def issuer():
        def issue_s(j):
            s = j % stages
            yield from sim.wait("kf%d" % s, j // stages)
            sim.mma(reads=("sQ", "sK%d" % s), writes=("S%d" % (j & 1),))
            sim.commit("s%d" % (j & 1), phase=j >> 1)
            sim.commit("ke%d" % s, phase=j // stages)
        yield from sim.wait("q", 0)
        yield from issue_s(0)
        if nsub > 1:
            yield from issue_s(1)
        for j in range(nsub):
            if plant == "one_p_barrier":
                yield from sim.work(0, 60)      # a slow issuer
            yield from sim.wait(P(j), Pk(j))
            s = j % stages
            yield from sim.wait("vf%d" % s, j // stages)
            sim.mma(reads=("sP%d" % (j & 1), "sV%d" % s), writes=("O",))
            sim.commit("o%d" % (j & 1), phase=j >> 1)
            sim.commit("ve%d" % s, phase=j // stages)
            if j + 2 < nsub:
                yield from issue_s(j + 2)

    def softmax():
        for j in range(nsub):
            yield from sim.wait("s%d" % (j & 1), j >> 1)
            t0 = sim.t
            yield from sim.work()
            if j > 0 and sim.rnd.random() < 0.3:   # a lazy rescale of O
                if plant != "rescale_unguarded":
                    yield from sim.wait("o%d" % ((j - 1) & 1), (j - 1) >> 1)
                t1 = sim.t
                yield from sim.work(1, 4)
                sim.touch("warp", "w", t1, "O")
            if j >= 2:
                yield from sim.wait("o%d" % (j & 1), (j - 2) >> 1)
            t2 = sim.t
            yield from sim.work(1, 4)
            sim.touch("warp", "w", t2, "sP%d" % (j & 1))
            sim.touch("warp", "r", t0, "S%d" % (j & 1))
            sim.arrive(P(j), phase=Pk(j))
        yield from sim.wait("o%d" % ((nsub - 1) & 1), (nsub - 1) >> 1)
        t3 = sim.t
        yield from sim.work(1, 4)
        sim.touch("warp", "r", t3, "O")

    sim.run([loader(), issuer()] + [softmax() for _ in range(nsoft)])
    return sim.errors


# -------------------------------------------------------------- dK / dV
def dkv(nsub, seed, plant=None, staged=True, ncomp=DKV_WARPS, stages=DKV_STAGES):
    """Loader warp: k, v once; q(j), dy(j) (and, staged, that sub-block's
    lse / D) into ring stage j % stages once dV, dK(j - stages) have read it;
    not staged, the whole block's lse / D by plain stores first.  MMA warp:
    S^T(j), dP^T(j) into tensor memory once the warps have copied out
    S^T(j - 1), dP^T(j - 1); then dV, dK(j - 1) from P^T, dS^T(j - 1).
    Compute warps: S^T, dP^T -> P^T, dS^T in tensor memory (after dV,
    dK(j - 1) have read them); dV, dK read at the end."""
    sim = Sim(seed, plant)
    for n in ("kv", "ld", "sf", "pe", "done"):
        sim.bar(n)
    for s in range(stages):
        sim.bar("qf%d" % s)
        sim.bar("qe%d" % s)
    sim.bar("se", ncomp)
    sim.bar("pf", ncomp)

    def stage_bufs(s):
        return ("sQ%d" % s, "sD%d" % s) + (("sLD%d" % s,) if staged else ())

    def loader():
        sim.tma("kv", "sK", "sV", phase=0)
        for j in range(min(nsub, stages)):
            sim.tma("qf%d" % (j % stages), *stage_bufs(j % stages), phase=0)
        if not staged:
            t0 = sim.t
            yield from sim.work(1, 6)
            sim.touch("loader", "w", t0, "sLD")
        sim.arrive("ld", phase=0)
        for j in range(stages, nsub):
            s = j % stages
            yield from sim.wait("qe%d" % s, j // stages - 1)
            sim.tma("qf%d" % s, *stage_bufs(s), phase=j // stages)

    def mma():
        yield from sim.wait("kv", 0)
        for j in range(nsub + 1):
            if j < nsub:
                s = j % stages
                yield from sim.wait("qf%d" % s, j // stages)
                if j > 0:
                    yield from sim.wait("se", j - 1)
                sim.mma(reads=("sK", "sV", "sQ%d" % s, "sD%d" % s), writes=("St", "dPt"))
                sim.commit("sf", phase=j)
            if j >= 1:
                jj = j - 1
                s = jj % stages
                yield from sim.wait("pf", jj)
                sim.mma(reads=("Pt", "dSt", "sQ%d" % s, "sD%d" % s), writes=("dV", "dK"))
                sim.commit("pe", phase=jj)
                sim.commit("qe%d" % s, phase=jj // stages)
        sim.commit("done", phase=0)

    def compute():
        yield from sim.wait("ld", 0)
        for j in range(nsub):
            s = j % stages
            yield from sim.wait("sf", j)
            t0 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "r", t0, "St", "dPt")
            sim.arrive("se", phase=j)
            if staged:  # the stage's lse / D arrive with its q / dy tiles
                yield from sim.wait("qf%d" % s, j // stages)
            t1 = sim.t
            yield from sim.work()
            if j > 0 and plant != "p_overwrite_unguarded":
                yield from sim.wait("pe", j - 1)
            t2 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "w", t2, "Pt", "dSt")
            sim.touch("warp", "r", t1, "sLD%d" % s if staged else "sLD")
            sim.arrive("pf", phase=j)
        yield from sim.wait("done", 0)
        t3 = sim.t
        yield from sim.work(1, 3)
        sim.touch("warp", "r", t3, "dV", "dK")

    sim.run([loader(), mma()] + [compute() for _ in range(ncomp)])
    return sim.errors


# -------------------------------------------------------------- dQ
def dq(nsub, seed, plant=None, ncomp=DQ_WARPS, kst=DQ_K_STAGES, vst=DQ_V_STAGES):
    """One warp loads and issues: q, dy once, k(0..kst-1), v(0..vst-1); S(0),
    dP(0).  Per sub-block j: once the warps have copied out S(j), dP(j),
    v(j + vst) into v's stage and S(j + 1), dP(j + 1); once dS(j) is in
    shared memory buffer j % 2, dQ(j); once dQ(j - 1) has read k's stage,
    k(j + 2) into it.  Compute warps: S(j), dP(j) -> dS(j) (after dQ(j - 2)
    has read the buffer); dQ read at the end."""
    sim = Sim(seed, plant)
    for n in ("q", "sf", "done"):
        sim.bar(n)
    for s in range(kst):
        sim.bar("kf%d" % s)
        sim.bar("ke%d" % s)
    for s in range(vst):
        sim.bar("vf%d" % s)
    sim.bar("se", ncomp)
    for i in range(2):
        sim.bar("pf%d" % i, ncomp)
        sim.bar("pe%d" % i)

    def issuer():
        def load_k(j):
            sim.tma("kf%d" % (j % kst), "sK%d" % (j % kst), phase=j // kst)

        def load_v(j):
            sim.tma("vf%d" % (j % vst), "sV%d" % (j % vst), phase=j // vst)

        def issue_sdp(j):
            ks, vs = j % kst, j % vst
            yield from sim.wait("kf%d" % ks, j // kst)
            yield from sim.wait("vf%d" % vs, j // vst)
            sim.mma(reads=("sQ", "sD", "sK%d" % ks, "sV%d" % vs), writes=("S", "dP"))
            sim.commit("sf", phase=j)
        sim.tma("q", "sQ", "sD", phase=0)
        for j in range(min(kst, nsub)):
            load_k(j)
        for j in range(min(vst, nsub)):
            load_v(j)
        yield from sim.wait("q", 0)
        yield from issue_sdp(0)
        for j in range(nsub):
            if j + 1 < nsub:
                yield from sim.wait("se", j)
                if j + vst < nsub:
                    load_v(j + vst)
                yield from issue_sdp(j + 1)
            yield from sim.wait("pf%d" % (j & 1), j >> 1)
            ks = j % kst
            sim.mma(reads=("sS%d" % (j & 1), "sK%d" % ks), writes=("dQ",))
            sim.commit("pe%d" % (j & 1), phase=j >> 1)
            sim.commit("ke%d" % ks, phase=j // kst)
            if j >= 1 and j + 2 < nsub:
                if plant != "k_refill_unguarded":
                    yield from sim.wait("ke%d" % ((j - 1) % kst), (j - 1) // kst)
                load_k(j + 2)
        sim.commit("done", phase=0)

    def compute():
        for j in range(nsub):
            yield from sim.wait("sf", j)
            t0 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "r", t0, "S", "dP")
            sim.arrive("se", phase=j)
            # dQ(j - 2) has read dS buffer j % 2; for j < 2 the wait is on
            # phase -1 (the barrier must still be in phase 0)
            k = (j - 2) >> 1 if plant != "p_wrong_phase" else j >> 1
            yield from sim.wait("pe%d" % (j & 1), k)
            t1 = sim.t
            yield from sim.work(1, 4)
            sim.touch("warp", "w", t1, "sS%d" % (j & 1))
            sim.arrive("pf%d" % (j & 1), phase=j >> 1)
        yield from sim.wait("done", 0)
        t2 = sim.t
        yield from sim.work(1, 3)
        sim.touch("warp", "r", t2, "dQ")

    sim.run([issuer()] + [compute() for _ in range(ncomp)])
    return sim.errors


NSUB = list(range(1, 10)) + [16, 17]


@pytest.mark.parametrize("model", [forward, dkv, dq])
def test_protocol_has_no_deadlock_aliased_wait_or_race(model):
    for nsub in NSUB:
        for seed in range(8):
            errs = model(nsub, seed)
            assert not errs, (model.__name__, nsub, seed, errs[:3])


def test_dkv_protocol_with_whole_block_lse_preload():
    for nsub in (1, 3, 5, 8):
        for seed in range(8):
            errs = dkv(nsub, seed, staged=False)
            assert not errs, (nsub, seed, errs[:3])


@pytest.mark.parametrize("model,plant,kind", [
    (forward, "one_p_barrier", "aliased wait"),
    (forward, "k_refill_unguarded", "race on sK"),
    (forward, "rescale_unguarded", "race on O"),
    (dkv, "p_overwrite_unguarded", "race on Pt"),
    (dq, "k_refill_unguarded", "race on sK"),
    (dq, "p_wrong_phase", "no progress"),
])
def test_the_checker_finds_a_planted_mistake(model, plant, kind):
    errs = find(model, plant, kind, range(4, 12))
    assert errs, "%s with %s: not found" % (model.__name__, plant)


# -------------------------------------------------------------- LayerNorm backward
LNB_STAGES = 2      # rows in flight per warp


def ln_bwd_ring(nrows, seed, plant=None, nwarps=3, stages=LNB_STAGES):
    """layernorm_bwd_kernel: warp w of nwarps takes rows w, w + nwarps, ...;
    its lane 0 bulk-copies the first `stages` of them (dy, x and the old
    residual gradient) into its own ring and, once the whole warp is done
    with a stage (__syncwarp), the row `stages` rows further on into it."""
    sim = Sim(seed, plant)

    def warp(w):
        for s in range(stages):
            sim.bar("b%d_%d" % (w, s))
        rows = list(range(w, nrows, nwarps))
        for i in range(min(stages, len(rows))):
            sim.tma("b%d_%d" % (w, i), "ring%d_%d" % (w, i), phase=0)
        for it, _ in enumerate(rows):
            s = it % stages
            yield from sim.wait("b%d_%d" % (w, s), it // stages)
            t0 = sim.t
            yield from sim.work(1, 4)
            if plant != "early_refill":
                sim.touch("lanes%d" % w, "r", t0, "ring%d_%d" % (w, s))
                yield                                   # __syncwarp: every lane is done with the stage
            else:                                       # no __syncwarp: a lane may still be reading
                sim.touch("lanes%d" % w, "r", t0, "ring%d_%d" % (w, s), until=sim.t + 3)
            if it + stages < len(rows):
                sim.tma("b%d_%d" % (w, s), "ring%d_%d" % (w, s), phase=(it + stages) // stages)

    sim.run([warp(w) for w in range(nwarps)])
    return sim.errors


def test_layernorm_backward_row_ring():
    for nrows in (1, 2, 5, 9, 20):
        for seed in range(6):
            errs = ln_bwd_ring(nrows, seed)
            assert not errs, (nrows, seed, errs[:3])
    assert find(ln_bwd_ring, "early_refill", "race on ring", [9, 20])
