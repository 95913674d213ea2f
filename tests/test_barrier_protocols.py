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
(csrc/k_attn_tc.cu), gemm_tc_pair_kernel (csrc/k_gemm_tc.cu) and
layernorm_bwd_kernel (csrc/k_misc.cu); a change
to a kernel's hand-offs changes its model.
"""
import pytest

from protocol_sim import Sim, find

# warps and ring stages as the kernels are compiled (head size 64): 8
# softmax warps, 2 query buffers and 2-stage key / value rings (forward);
# 16 elementwise warps, 2 key/value buffers and a 3-stage query ring
# (dK/dV); 16 elementwise warps, 2 query buffers, 5 key and 3 value stages
# (dQ).  A CTA walks a list of work items; ITEMS are the item lengths (key
# or query blocks) of the lists tried, longest first as the kernels order
# them.
FWD_WARPS, FWD_QB, FWD_KV = 8, 2, 2
DKV_WARPS, DKV_KVB, DKV_STAGES = 16, 2, 3
DQ_WARPS, DQ_QB, DQ_KST, DQ_VST = 16, 2, 5, 3
ITEMS = [[1], [3], [8, 5, 2], [4, 4, 1, 1], [2, 1, 1, 1, 1], [16, 9]]


# -------------------------------------------------------------- forward
def forward(items, seed, plant=None, nsoft=FWD_WARPS, qb=FWD_QB, kv=FWD_KV):
    """attn_fwd_tc_kernel.  Loader: per item q into buffer it % qb once the
    item qb back has issued its last S; per block k, v into ring stage
    g % kv once S(g - kv), PV(g - kv) have read it.  MMA issuer, over the
    blocks g of all items in turn: S(g) once k(g) is in and the softmax
    warps have copied S(g - 1) out; then PV(g - 1) once P(g - 1) is
    written (so PV of an item's last block runs after the next item's
    first S).  Softmax warps: copy S(g) out, then P(g) into tensor memory
    once PV(g - 1) has read the P columns (at an item's first block the
    previous item's epilogue has waited for that), with an occasional
    rescale of O in tensor memory at the same point; O read at the end of
    each item."""
    sim = Sim(seed, plant)
    for i in range(qb):
        sim.bar("qf%d" % i)
        sim.bar("qe%d" % i)
    for s in range(kv):
        for n in ("kf%d", "ke%d", "vf%d", "ve%d"):
            sim.bar(n % s)
    sim.bar("sf")
    sim.bar("sfree", nsoft)
    sim.bar("pf", nsoft)
    sim.bar("od")

    def loader():
        g = 0
        for it, nk in enumerate(items):
            qs = it % qb
            if it >= qb and plant != "q_refill_unguarded":
                yield from sim.wait("qe%d" % qs, it // qb - 1)
            sim.tma("qf%d" % qs, "sQ%d" % qs, phase=it // qb)
            for _ in range(nk):
                s = g % kv
                if g >= kv:
                    yield from sim.wait("ke%d" % s, g // kv - 1)
                sim.tma("kf%d" % s, "sK%d" % s, phase=g // kv)
                if g >= kv:
                    yield from sim.wait("ve%d" % s, g // kv - 1)
                sim.tma("vf%d" % s, "sV%d" % s, phase=g // kv)
                g += 1

    def issuer():
        def pv(gp, first):
            yield from sim.wait("pf", gp)
            yield from sim.wait("vf%d" % (gp % kv), gp // kv)
            sim.mma(reads=("P", "sV%d" % (gp % kv)) + (() if first else ("O",)), writes=("O",))
            sim.commit("ve%d" % (gp % kv), phase=gp // kv)
            sim.commit("od", phase=gp)
        g, prev = 0, None
        for it, nk in enumerate(items):
            qs = it % qb
            yield from sim.wait("qf%d" % qs, it // qb)
            for j in range(nk):
                yield from sim.wait("kf%d" % (g % kv), g // kv)
                if g > 0:
                    yield from sim.wait("sfree", g - 1)
                sim.mma(reads=("sQ%d" % qs, "sK%d" % (g % kv)), writes=("S",))
                sim.commit("ke%d" % (g % kv), phase=g // kv)
                if j == nk - 1:
                    sim.commit("qe%d" % qs, phase=it // qb)
                sim.commit("sf", phase=g)
                if prev is not None:
                    yield from pv(*prev)
                prev = (g, j == 0)
                g += 1
        if prev is not None:
            yield from pv(*prev)

    def softmax():
        g = 0
        for nk in items:
            for j in range(nk):
                yield from sim.wait("sf", g)
                t0 = sim.t
                yield from sim.work(1, 3)
                if plant == "s_free_early":
                    sim.arrive("sfree", phase=g)
                    yield from sim.work(1, 3)
                    sim.touch("warp", "r", t0, "S")
                else:
                    sim.touch("warp", "r", t0, "S")
                    sim.arrive("sfree", phase=g)
                yield from sim.work()
                if j > 0:
                    if plant != "p_unguarded":
                        yield from sim.wait("od", g - 1)
                    if sim.rnd.random() < 0.3:   # a lazy rescale of O
                        t1 = sim.t
                        yield from sim.work(1, 3)
                        sim.touch("warp", "w", t1, "O")
                t2 = sim.t
                yield from sim.work(1, 3)
                sim.touch("warp", "w", t2, "P")
                sim.arrive("pf", phase=g)
                g += 1
            yield from sim.wait("od", g - 1)
            t3 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "r", t3, "O")

    sim.run([loader(), issuer()] + [softmax() for _ in range(nsoft)])
    return sim.errors


# -------------------------------------------------------------- dK / dV
def dkv(items, seed, plant=None, staged=True, ncomp=DKV_WARPS, kvb=DKV_KVB, stages=DKV_STAGES):
    """attn_bwd_dkv_tc_kernel.  Loader: per item k, v into buffer it % kvb
    once the item kvb back has issued its last S^T, dP^T; per query
    sub-block g q, dy (and, staged, their lse / D) into ring stage
    g % stages once dV, dK(g - stages) have read it.  Every sub-block is
    taken in two column halves with their own hand-offs.  Score issuer, over
    all sub-blocks and halves in turn: S^T, dP^T (g, h) once group h has
    copied out its half of g - 1.  Gradient issuer (another thread, its MMAs
    interleave with the score issuer's in any order): dV, dK (g, h) from
    P^T, dS^T (g, h), half 0 before half 1; the first of an item overwrites
    the accumulators, its last commits their completion.
    Elementwise warps, two groups (group h owns half h): copy the half of
    S^T, dP^T out in two pieces, (staged) wait for the stage's lse / D, write
    P^T, dS^T once dV, dK (g - 1, h) have read them.  An item's dV, dK are
    read by group 0, one item late, in the next item's first sub-block
    before its half-0 products are released (and the last item's after the
    loop)."""
    sim = Sim(seed, plant)
    gw = ncomp // 2
    for i in range(kvb):
        sim.bar("kvf%d" % i)
        sim.bar("kve%d" % i)
    for s in range(stages):
        sim.bar("qf%d" % s)
        sim.bar("qe%d" % s)
    for h in range(2):
        sim.bar("sf%d" % h)
        sim.bar("sfree%d" % h, gw)
        sim.bar("pf%d" % h, gw)
        sim.bar("pe%d" % h)
    sim.bar("acc")

    def stage_bufs(s):
        return ("sQ%d" % s, "sD%d" % s) + (("sLD%d" % s,) if staged else ())

    def loader():
        g = 0
        for it, nsub in enumerate(items):
            b = it % kvb
            if it >= kvb and plant != "kv_refill_unguarded":
                yield from sim.wait("kve%d" % b, it // kvb - 1)
            sim.tma("kvf%d" % b, "sK%d" % b, "sV%d" % b, phase=it // kvb)
            for _ in range(nsub):
                s = g % stages
                if g >= stages:
                    yield from sim.wait("qe%d" % s, g // stages - 1)
                sim.tma("qf%d" % s, *stage_bufs(s), phase=g // stages)
                g += 1

    def score_mma():
        g = 0
        for it, nsub in enumerate(items):
            b = it % kvb
            yield from sim.wait("kvf%d" % b, it // kvb)
            for j in range(nsub):
                s = g % stages
                yield from sim.wait("qf%d" % s, g // stages)
                for h in range(2):
                    if g > 0:
                        yield from sim.wait("sfree%d" % h, g - 1)
                    sim.mma(reads=("sK%d" % b, "sV%d" % b, "sQ%d" % s, "sD%d" % s),
                            writes=("St%d" % h, "dPt%d" % h))
                    if h == 1 and j == nsub - 1:
                        sim.commit("kve%d" % b, phase=it // kvb)
                    sim.commit("sf%d" % h, phase=g)
                g += 1

    def grad_mma():
        g = 0
        for it, nsub in enumerate(items):
            for j in range(nsub):
                s = g % stages
                for h in range(2):
                    yield from sim.wait("pf%d" % h, g)
                    acc = () if (j == 0 and h == 0) else ("dV", "dK")
                    sim.mma(reads=("Pt%d" % h, "dSt%d" % h, "sQ%d" % s, "sD%d" % s) + acc, writes=("dV", "dK"))
                    sim.commit("pe%d" % h, phase=g)
                    if h == 1:
                        sim.commit("qe%d" % s, phase=g // stages)
                    if h == 1 and j == nsub - 1:
                        sim.commit("acc", phase=it)
                g += 1

    def compute(h):
        g = 0
        for it, nsub in enumerate(items):
            for j in range(nsub):
                s = g % stages
                yield from sim.wait("sf%d" % h, g)
                # two pieces: each read, computed and written before the next
                t0 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "r", t0, "St%d" % h, "dPt%d" % h)
                if staged:  # the stage's lse / D arrive with its q / dy tiles
                    yield from sim.wait("qf%d" % s, g // stages)
                t1 = sim.t
                yield from sim.work()
                if staged:
                    sim.touch("warp", "r", t1, "sLD%d" % s)
                if g > 0 and plant != "p_overwrite_unguarded":
                    yield from sim.wait("pe%d" % h, g - 1)
                t2 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "w", t2, "Pt%d" % h, "dSt%d" % h)
                t3 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "r", t3, "St%d" % h, "dPt%d" % h)
                sim.arrive("sfree%d" % h, phase=g)
                t4 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "w", t4, "Pt%d" % h, "dSt%d" % h)
                epi = h == 0 and j == 0 and it > 0
                if epi and plant != "epi_late":
                    # the previous item's dV, dK read before this item's
                    # first gradient products overwrite them
                    yield from sim.wait("acc", it - 1)
                    t5 = sim.t
                    yield from sim.work(1, 2)
                    sim.touch("warp", "r", t5, "dV", "dK")
                sim.arrive("pf%d" % h, phase=g)
                if epi and plant == "epi_late":
                    yield from sim.wait("acc", it - 1)
                    t5 = sim.t
                    yield from sim.work(1, 2)
                    sim.touch("warp", "r", t5, "dV", "dK")
                g += 1
        if h == 0 and items:  # the last item's accumulators
            yield from sim.wait("acc", len(items) - 1)
            t6 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "r", t6, "dV", "dK")

    sim.run([loader(), score_mma(), grad_mma()] + [compute(w // gw) for w in range(ncomp)])
    return sim.errors


# -------------------------------------------------------------- dQ
def dq(items, seed, plant=None, ncomp=DQ_WARPS, qb=DQ_QB, kst=DQ_KST, vst=DQ_VST):
    """attn_bwd_dq_tc_kernel.  Loader: per item q, dy into buffer it % qb
    once the item qb back has issued its last S, dP; per key block k into
    stage g % kst once dQ(g - kst) has read it, v into stage g % vst once
    dP(g - vst) has.  Every block is taken in two key halves with their own
    hand-offs.  Score issuer, over all blocks and halves in turn: S, dP
    (g, h) once group h has copied out its half of g - 1.  dQ issuer
    (another thread): dQ from dS (g, h), half 0 before half 1; the first of
    an item overwrites dQ, its last commits dQ's completion.
    Elementwise warps, two groups (group h owns half h): copy the half of S,
    dP out in two pieces, write its dS once dQ (g - 1, h) has read it.  An
    item's dQ is read by group 0, one item late, in the next item's first
    block before its half-0 products are released (and the last item's
    after the loop)."""
    sim = Sim(seed, plant)
    gw = ncomp // 2
    for i in range(qb):
        sim.bar("qf%d" % i)
        sim.bar("qe%d" % i)
    for s in range(kst):
        sim.bar("kf%d" % s)
        sim.bar("ke%d" % s)
    for s in range(vst):
        sim.bar("vf%d" % s)
        sim.bar("ve%d" % s)
    for h in range(2):
        sim.bar("sf%d" % h)
        sim.bar("sfree%d" % h, gw)
        sim.bar("pf%d" % h, gw)
        sim.bar("dsf%d" % h)
    sim.bar("dqf")

    def loader():
        g = 0
        for it, nk in enumerate(items):
            b = it % qb
            if it >= qb:
                yield from sim.wait("qe%d" % b, it // qb - 1)
            sim.tma("qf%d" % b, "sQ%d" % b, "sD%d" % b, phase=it // qb)
            for _ in range(nk):
                ks, vs = g % kst, g % vst
                if g >= kst and plant != "k_refill_unguarded":
                    yield from sim.wait("ke%d" % ks, g // kst - 1)
                sim.tma("kf%d" % ks, "sK%d" % ks, phase=g // kst)
                if g >= vst:
                    yield from sim.wait("ve%d" % vs, g // vst - 1)
                sim.tma("vf%d" % vs, "sV%d" % vs, phase=g // vst)
                g += 1

    def score_mma():
        g = 0
        for it, nk in enumerate(items):
            b = it % qb
            yield from sim.wait("qf%d" % b, it // qb)
            for j in range(nk):
                ks, vs = g % kst, g % vst
                yield from sim.wait("kf%d" % ks, g // kst)
                yield from sim.wait("vf%d" % vs, g // vst)
                for h in range(2):
                    if g > 0:
                        yield from sim.wait("sfree%d" % h, g - 1)
                    sim.mma(reads=("sQ%d" % b, "sD%d" % b, "sK%d" % ks, "sV%d" % vs), writes=("S%d" % h, "dP%d" % h))
                    if h == 1:
                        sim.commit("ve%d" % vs, phase=g // vst)
                        if j == nk - 1:
                            sim.commit("qe%d" % b, phase=it // qb)
                    sim.commit("sf%d" % h, phase=g)
                g += 1

    def dq_mma():
        g = 0
        for it, nk in enumerate(items):
            for j in range(nk):
                ks = g % kst
                for h in range(2):
                    k = g if plant != "ds_wrong_phase" else g + 1
                    yield from sim.wait("pf%d" % h, k)
                    sim.mma(reads=("dS%d" % h, "sK%d" % ks) + (() if (j == 0 and h == 0) else ("dQ",)), writes=("dQ",))
                    sim.commit("dsf%d" % h, phase=g)
                    if h == 1:
                        sim.commit("ke%d" % ks, phase=g // kst)
                        if j == nk - 1:
                            sim.commit("dqf", phase=it)
                g += 1

    def compute(h):
        g = 0
        for it, nk in enumerate(items):
            for j in range(nk):
                yield from sim.wait("sf%d" % h, g)
                # two pieces: each read, computed and its dS written before the next
                t0 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "r", t0, "S%d" % h, "dP%d" % h)
                yield from sim.work()
                if g > 0:
                    yield from sim.wait("dsf%d" % h, g - 1)
                t1 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "w", t1, "dS%d" % h)
                t2 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "r", t2, "S%d" % h, "dP%d" % h)
                sim.arrive("sfree%d" % h, phase=g)
                t3 = sim.t
                yield from sim.work(1, 2)
                sim.touch("warp", "w", t3, "dS%d" % h)
                if h == 0 and j == 0 and it > 0:
                    # the previous item's dQ read before this item's first
                    # dQ products overwrite it
                    yield from sim.wait("dqf", it - 1)
                    t4 = sim.t
                    yield from sim.work(1, 2)
                    sim.touch("warp", "r", t4, "dQ")
                sim.arrive("pf%d" % h, phase=g)
                g += 1
        if h == 0 and items:  # the last item's dQ
            yield from sim.wait("dqf", len(items) - 1)
            t5 = sim.t
            yield from sim.work(1, 3)
            sim.touch("warp", "r", t5, "dQ")

    sim.run([loader(), score_mma(), dq_mma()] + [compute(w // gw) for w in range(ncomp)])
    return sim.errors


@pytest.mark.parametrize("model", [forward, dkv, dq])
def test_protocol_has_no_deadlock_aliased_wait_or_race(model):
    for items in ITEMS:
        for seed in range(6):
            errs = model(items, seed)
            assert not errs, (model.__name__, items, seed, errs[:3])


def test_protocols_with_one_buffer_per_item_and_head_size_128_rings():
    # head size 128: one q buffer (forward keeps two), one k/v buffer set
    # (dK/dV), one q/dy buffer and 2 key stages (dQ)
    for items in ITEMS:
        for seed in range(4):
            assert not dkv(items, seed, kvb=1), items
            assert not dq(items, seed, qb=1, kst=2), items
            assert not forward(items, seed, qb=1), items


def test_dkv_protocol_with_lse_and_d_from_global_memory():
    for items in ITEMS:
        for seed in range(4):
            errs = dkv(items, seed, staged=False)
            assert not errs, (items, seed, errs[:3])


def _find(model, plant, kind, seeds=12, **kw):
    for items in ITEMS[2:]:
        for seed in range(seeds):
            errs = model(items, seed, plant=plant, **kw)
            if any(kind in e for e in errs):
                return errs
    return []


@pytest.mark.parametrize("model,plant,kind,kw", [
    (forward, "s_free_early", "race on S", {}),
    (forward, "p_unguarded", "race on P", {}),
    (forward, "q_refill_unguarded", "race on sQ", dict(qb=1)),
    (dkv, "p_overwrite_unguarded", "race on Pt", {}),
    (dkv, "kv_refill_unguarded", "race on sK", dict(kvb=1)),
    (dkv, "epi_late", "race on dV", {}),
    (dq, "k_refill_unguarded", "race on sK", dict(kst=2)),
    (dq, "ds_wrong_phase", "no progress", {}),
])
def test_the_checker_finds_a_planted_mistake(model, plant, kind, kw):
    errs = _find(model, plant, kind, **kw)
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


# -------------------------------------------------------------- matmul CTA pairs
GEMM_STAGES = 6


def gemm_pair(ntiles, seed, plant=None, stages=GEMM_STAGES, kt=3):
    """gemm_tc_pair_kernel: CTA r of the pair loads its A rows and its half
    of the B tile into stage s; every byte lands on the leader's full[s]
    (the leader's arrive.expect_tx is one more arrival).  The leader's MMA
    thread issues a tile's k steps into accumulator a = tile % 2 once both
    CTAs' epilogues released it, and its commits release stage s in both
    CTAs (empty[s]) and hand the accumulator to both epilogues."""
    sim = Sim(seed, plant)
    for st in range(stages):
        sim.bar("full_%d" % st, 5)  # expect + 2 A loads + 2 B halves
        for c in range(2):
            sim.bar("empty%d_%d" % (c, st))
    for a in range(2):
        sim.bar("accf_%d" % a)
        sim.bar("acce_%d" % a, 2)
    nsteps = ntiles * kt

    def producer(c):
        for it in range(nsteps):
            st, ph = it % stages, it // stages
            if it >= stages and plant != "refill_unguarded":
                yield from sim.wait("empty%d_%d" % (c, st), ph - 1)
            if c == 0:
                sim.arrive("full_%d" % st, ph)
            sim.tma("full_%d" % st, "A%d_%d" % (c, st), phase=ph)
            sim.tma("full_%d" % st, "B%d_%d" % (c, st), phase=ph)
            yield from sim.work(0, 2)
        for d in range(max(0, nsteps - stages), nsteps):  # the last releases have landed
            yield from sim.wait("empty%d_%d" % (c, d % stages), d // stages)

    def issuer():
        it = 0
        for ti in range(ntiles):
            a = ti & 1
            if ti >= 2:
                yield from sim.wait("acce_%d" % a, ti // 2 - 1)
            for _ in range(kt):
                st, ph = it % stages, it // stages
                yield from sim.wait("full_%d" % st, ph)
                reads = ["A%d_%d" % (c, st) for c in range(2)] + ["B%d_%d" % (c, st) for c in range(2)]
                sim.mma(reads=reads, writes=["acc_%d" % a])
                for c in range(2):
                    sim.commit("empty%d_%d" % (c, st), ph)
                it += 1
                yield
            sim.commit("accf_%d" % a, ti // 2)
        for d in range(max(0, ntiles - 2), ntiles):
            yield from sim.wait("acce_%d" % (d & 1), d // 2)

    def epilogue(c):
        for ti in range(ntiles):
            a = ti & 1
            yield from sim.wait("accf_%d" % a, ti // 2)
            t0 = sim.t
            yield from sim.work(1, 12)
            if plant == "acc_release_early":  # released before the last TMEM loads are done
                sim.arrive("acce_%d" % a, ti // 2)
                sim.touch("epi%d" % c, "r", t0, "acc_%d" % a, until=sim.t + 100)
            else:
                sim.touch("epi%d" % c, "r", t0, "acc_%d" % a)
                sim.arrive("acce_%d" % a, ti // 2)

    sim.run([producer(c) for c in range(2)] + [issuer()] + [epilogue(c) for c in range(2)])
    return sim.errors


def test_matmul_pair_protocol():
    for ntiles in (1, 2, 3, 7):
        for kt in (1, 2, 5, 12):
            for seed in range(3):
                errs = gemm_pair(ntiles, seed, kt=kt)
                assert not errs, (ntiles, kt, seed, errs[:3])
    for seed in range(3):
        assert not gemm_pair(5, seed, stages=2, kt=3)


@pytest.mark.parametrize("plant,kind", [
    ("refill_unguarded", "race on A"),     # a stage refilled while the MMAs still read it
    ("acc_release_early", "race on acc"),  # the accumulator handed back before it is read out
])
def test_matmul_pair_checker_finds_a_planted_mistake(plant, kind):
    assert find(lambda n, seed, plant=None: gemm_pair(n, seed, plant=plant, stages=2, kt=1),
                plant, kind, [3, 7], seeds=12)
