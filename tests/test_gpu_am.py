"""GPU parity of Attention Matching (the bias beta and compact values V_C fitted on the survivors)
with the oracle.

Source: "Practical Online KV Cache Compaction for LLM Agents: An Empirical Study" (agifrontier
tutorial page), section on the two compaction families: min ||exp(Q K_C^T + beta) 1_m -
exp(Q K^T) 1_n||^2 and min ||A_hat(Q; K_C, beta, V_C) - A(Q; K, V)||_F^2.

What is compared depends on how well the unit's problem is conditioned:

* Well-conditioned units (cond(E) <= 1e8: diffuse or aligned proxy queries): the residual norm
  each fit reaches after the same sweeps, evaluated in fp64 by the oracle on its own problem
  (E, s, Y) at the GPU's outputs, must equal the oracle's own to RES_TOL = 1e-5 of the target
  norm (mass: |s|; value: |Y|).  Derivation: the GPU forms E and s from fp32 logits (128-term
  fp32 dot products: relative error ~1e-6 on diffuse rows), the Gram matrices over R rows and
  the descent in fp32, and freezes coordinates whose gradient is below 2^-17 of its terms'
  scale; on every unit of these cases and of the multi-turn shape's three query recipes the
  measured gap is at most 5.4e-6; the bound leaves a factor of ~2.
  Where R > m and the fit is small, w and V_C themselves are compared element by element,
  against a per-unit bound the oracle derives: it re-runs both fits with E, s and Y perturbed by
  independent relative noise of EPS = 1e-5 (a few times the rounding the GPU's inputs to the
  fits carry: fp32-accumulated logits, the probabilities held as two bf16 parts, the LSE
  normalisation) and takes the largest change of w (relative to max(1, |w|)) and of V_C
  (relative to max |V_C|) over ENV_DRAWS draws; the GPU's w and V_C must lie within ENV_FACTOR
  times that envelope of the oracle's.  After 8 sweeps V_C moves by up to ~100x the input noise
  on these units (the descent has not converged and Ph is not well conditioned), so a fixed
  bound would measure the fit's conditioning rather than the kernel.
* Concentrated units (cond(E) > 1e8, up to 1e18 with planted proxy queries): the gradient of a
  key with almost no attention is rounding in any precision, and the plain fp64 descent itself
  takes steps of that size (w_j to 1e3), after which its value residual can stand above token
  eviction's.  Neither side's value fit is unique there.  The mass residual is still compared
  two-sided at RES_TOL; the GPU's value residual must not exceed the oracle's by more than
  RES_TOL (it may be lower).  Without the kernel's rounding guard an fp32 descent diverges on
  these units (value residual 1e-2 of |Y| above the oracle's), which this check catches.

The keep sets come from the oracle's own token-eviction scores, and every value the tests
expect comes from the oracle.
"""
import numpy as np
import pytest
import torch

import online_kv_cache_gb300 as kvc
import oracle
import workloads
from oracle import am
from tests import parity as PT

pytestmark = pytest.mark.gpu
DEV = "cuda"
RES_TOL = 1e-5
EPS = 1e-5
ENV_DRAWS = 6
ENV_FACTOR = 3.0
COND_WELL = 1e8


@pytest.fixture(scope="module", autouse=True)
def built():
    from online_kv_cache_gb300 import build
    build.build()
    kvc.kvc_read_device_status(clear=True)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_keep(case, m):
    s, _ = oracle.score_cache(case.k_pool, case.block_table, case.nblocks, case.seg_start, case.seg_end,
                              case.seq_len, case.q, case.spec.scale)
    return oracle.select_cache(s, case.seg_start, case.seg_end, m)


def run_gpu(case, m, keep_np, sweeps, aux):
    sp = case.spec
    cp = kvc.Compactor(case.k_pool, case.v_pool, case.tags, case.block_table, case.nblocks, case.free_ids,
                       case.free_top, case.seg_start, case.seg_end, case.seq_len, m, sp.R, aux=aux)
    keep = torch.from_numpy(np.ascontiguousarray(keep_np)).to(DEV)
    beta = torch.full((sp.L, sp.H, max(1, cp.Mtot)), float("nan"), device=DEV)
    vc = torch.full((sp.L, sp.H, max(1, cp.Mtot), sp.d), float("nan"), device=DEV)
    cp.am_fit(case.q, sp.scale, sweeps, keep=keep, beta=beta, vc=vc)
    torch.cuda.synchronize()
    PT.device_status_clean()
    return beta.cpu().numpy().astype(np.float64), vc.cpu().numpy().astype(np.float64)


def envelope(u, sweeps, key):
    """Largest change of the oracle's w and V_C when its inputs E, s and Y carry independent
    relative noise of EPS (seeded per unit)."""
    rng = np.random.default_rng(abs(hash(key)) % (2 ** 32))
    X0 = u["x0"]
    ew = ev = 0.0
    for _ in range(ENV_DRAWS):
        E = u["E"] * (1 + EPS * rng.standard_normal(u["E"].shape))
        s = u["s"] * (1 + EPS * rng.standard_normal(u["s"].shape))
        Y = u["Y"] * (1 + EPS * rng.standard_normal(u["Y"].shape))
        w = am.mass_fit(E, s, sweeps)
        X = am.value_fit(am.compact_probs(E, w), Y, X0, sweeps)
        ew = max(ew, np.max(np.abs(w - u["w"]) / np.maximum(1.0, np.abs(u["w"]))))
        ev = max(ev, np.max(np.abs(X - u["vc"])) / np.abs(u["vc"]).max())
    return ew, ev


def check_units(units, m, beta, vc, sweeps, sample=None, elementwise=False):
    """Residuals of both fits at the GPU's outputs against the oracle's, per unit (two-sided on
    well-conditioned units, one-sided for the value fit on concentrated ones); w and V_C element
    by element when asked."""
    moff = np.concatenate([[0], np.cumsum(m)])
    worst = {"mass": 0.0, "value": 0.0, "value_excess": 0.0, "w": 0.0, "vc": 0.0}
    kinds = {"well": 0, "concentrated": 0}
    keys = sorted(units) if sample is None else sample
    for (b, l, h) in keys:
        u = units[(b, l, h)]
        sl = slice(moff[b], moff[b + 1])
        bg = beta[l, h, sl]
        assert not np.any(np.isnan(bg)) and not np.any(bg == np.inf)
        assert np.all(np.isfinite(vc[l, h, sl]))
        wg = np.exp(bg)  # exp(-inf) = 0: a masked key
        well = u["E"].shape[1] == 0 or np.linalg.cond(u["E"]) <= COND_WELL
        kinds["well" if well else "concentrated"] += 1
        s_norm = np.linalg.norm(u["s"])
        r_gpu = np.sqrt(am.mass_objective(u["E"], u["s"], wg))
        r_orc = np.sqrt(am.mass_objective(u["E"], u["s"], u["w"]))
        dm = abs(r_gpu - r_orc) / s_norm
        assert dm <= RES_TOL, f"unit {(b, l, h)}: mass residual {r_gpu:.4e} vs oracle {r_orc:.4e} (|s| {s_norm:.3e})"
        y_norm = np.linalg.norm(u["Y"])
        v_gpu = np.sqrt(am.value_objective(u["E"], u["Y"], wg, vc[l, h, sl]))
        v_orc = np.sqrt(am.value_objective(u["E"], u["Y"], u["w"], u["vc"]))
        if well:
            dv = abs(v_gpu - v_orc) / y_norm
            assert dv <= RES_TOL, f"unit {(b, l, h)}: value residual {v_gpu:.4e} vs oracle {v_orc:.4e} (|Y| {y_norm:.3e})"
            worst["value"] = max(worst["value"], dv)
        else:
            ex = (v_gpu - v_orc) / y_norm
            assert ex <= RES_TOL, f"unit {(b, l, h)}: value residual {v_gpu:.4e} above the oracle's {v_orc:.4e} (|Y| {y_norm:.3e})"
            worst["value_excess"] = max(worst["value_excess"], ex)
        worst["mass"] = max(worst["mass"], dm)
        if elementwise and u["E"].shape[1] > 0:
            assert well
            env_w, env_v = envelope(u, sweeps, (b, l, h))
            ew = np.max(np.abs(wg - u["w"]) / np.maximum(1.0, np.abs(u["w"])))
            ev = np.max(np.abs(vc[l, h, sl] - u["vc"])) / np.abs(u["vc"]).max()
            assert ew <= ENV_FACTOR * env_w + 1e-7, \
                f"unit {(b, l, h)}: w differs by {ew:.3e} of max(1, |w|) (envelope {env_w:.3e})"
            assert ev <= ENV_FACTOR * env_v + 1e-7, \
                f"unit {(b, l, h)}: V_C differs by {ev:.3e} of max |V_C| (envelope {env_v:.3e})"
            worst["w"], worst["vc"] = max(worst["w"], ew / (env_w + 1e-12)), max(worst["vc"], ev / (env_v + 1e-12))
    print(f"sweeps={sweeps} units {kinds}: worst gaps " + ", ".join(f"{k} {v:.2e}" for k, v in worst.items())
          + " (w, vc: in units of the unit's envelope)")
    return kinds


def check_writes(case, m, keep_np, beta, vc, before_v, before_k, before_aux, aux):
    """Kept V rows hold bf16(V_C) (round to nearest even), their aux slots hold beta; every other
    V row, every K row and every other aux slot is untouched."""
    sp = case.spec
    v_after = case.v_pool.cpu()
    k_after = case.k_pool.cpu()
    assert torch.equal(k_after, before_k)
    bt = case.block_table.cpu().numpy()
    moff = np.concatenate([[0], np.cumsum(m)])
    want_v = before_v.clone()
    want_aux = before_aux.copy()
    for b in range(sp.B):
        for l in range(sp.L):
            for h in range(sp.H):
                for j in range(m[b]):
                    pos = int(keep_np[l, h, moff[b] + j])
                    slot = case.seg_start[b] + pos
                    pg, o = bt[b, slot // sp.P], slot % sp.P
                    want_v[l, pg, h, o] = torch.from_numpy(vc[l, h, moff[b] + j].astype(np.float32)).to(torch.bfloat16)
                    want_aux[l, pg, h, o] = beta[l, h, moff[b] + j]
    assert torch.equal(v_after.view(torch.int16), want_v.view(torch.int16))
    got_aux = aux.cpu().numpy()
    assert np.array_equal(np.isneginf(got_aux), np.isneginf(want_aux))
    fin = np.isfinite(want_aux)
    assert np.array_equal(got_aux[fin], want_aux[fin].astype(np.float32))


@pytest.mark.parametrize("d,P,G,q,lengths,ratio,sweeps,qdist,elementwise", [
    (128, 16, 4, 8, (300, 129), 0.2, 8, "planted4", False),  # R = 32 < m, concentrated (cond(E) ~1e15)
    (128, 16, 4, 8, (300, 129), 0.2, 8, "normal", False),    # diffuse attention, m > R: many minimisers
    (64, 32, 2, 40, (200, 65, 1), 0.2, 8, "normal", True),   # R = 80 > m, a one-key unit: w, V_C compared
    (64, 16, 4, 32, (160, 97), 0.2, 8, "normal", True),      # R = 128 > m, two sequences
    (128, 16, 8, 16, (700,), 0.1, 3, "aligned", False),      # Q-aligned heavy hitters, two key tiles of rows
    # m = 640 and 300 in one launch (laid out for the larger): five row tiles of the Gram products,
    # blocks whose three tiles span two tile rows and read four strips, G's column m alone in a
    # sixth column tile
    (64, 16, 2, 48, (3200, 1500), 0.2, 8, "normal", False),
    # R = 8: one 16-row chunk, so Ph^T Y is summed over one row range (R = 32, 80, 96 and 128
    # above give two, four uneven and four even ranges)
    (64, 16, 2, 4, (120, 40), 0.2, 8, "normal", False),
])
def test_am_matches_oracle(d, P, G, q, lengths, ratio, sweeps, qdist, elementwise):
    sp = workloads.custom(L=2, H=2, G=G, d=d, P=P, q=q, lengths=lengths, shuffle_pages=True,
                          qdist=qdist)
    case = workloads.build(sp, 5, DEV)
    m = [oracle.budget_ratio(n, ratio) for n in PT.seg_lengths(case)]
    keep_np = oracle_keep(case, m)
    g = torch.Generator(device=DEV).manual_seed(3)
    aux = torch.rand(case.tags.shape, generator=g, device=DEV)
    before = (case.v_pool.cpu().clone(), case.k_pool.cpu().clone(), aux.cpu().numpy().copy())
    kb, vb, qb = bits(case.k_pool), bits(case.v_pool), bits(case.q)
    beta, vc = run_gpu(case, m, keep_np, sweeps, aux)
    _, _, units = am.cache(kb, vb, qb, case.block_table.cpu().numpy(), case.seg_start, case.seg_end, keep_np, m,
                           sp.scale, sweeps)
    kinds = check_units(units, m, beta, vc, sweeps, elementwise=elementwise)
    if qdist == "planted4":
        assert kinds["concentrated"] > 0  # the regime the guard is for
    else:
        assert kinds["concentrated"] == 0
    check_writes(case, m, keep_np, beta, vc, *before, aux)


def test_zero_sweeps_is_token_eviction():
    """sweeps = 0 returns token eviction's answer: beta = 0, V_C = V, the pool unchanged."""
    sp = workloads.custom(L=1, H=2, G=2, d=128, P=16, q=8, lengths=(257,), shuffle_pages=True)
    case = workloads.build(sp, 6, DEV)
    m = [oracle.budget_ratio(257, 0.2)]
    keep_np = oracle_keep(case, m)
    v0 = case.v_pool.cpu().clone()
    beta, vc = run_gpu(case, m, keep_np, 0, None)
    assert np.all(beta == 0.0)
    assert torch.equal(case.v_pool.cpu().view(torch.int16), v0.view(torch.int16))
    _, _, units = am.cache(bits(case.k_pool), bits(case.v_pool), bits(case.q), case.block_table.cpu().numpy(),
                           case.seg_start, case.seg_end, keep_np, m, sp.scale, 0)
    for (b, l, h), u in units.items():
        np.testing.assert_array_equal(vc[l, h, :m[0]], u["vc"])  # the bf16 values, exactly


def test_keep_all_reproduces_the_full_attention():
    """m = n: the kept keys carry all the mass and V reproduces the output; the fits stay at
    (numerically) zero residual."""
    sp = workloads.custom(L=1, H=2, G=4, d=64, P=16, q=8, lengths=(96,))
    case = workloads.build(sp, 7, DEV)
    m = [96]
    keep_np = np.tile(np.arange(96, dtype=np.int32), (1, 2, 1))
    beta, vc = run_gpu(case, m, keep_np, 4, None)
    _, _, units = am.cache(bits(case.k_pool), bits(case.v_pool), bits(case.q), case.block_table.cpu().numpy(),
                           case.seg_start, case.seg_end, keep_np, m, sp.scale, 4)
    check_units(units, m, beta, vc, 4)
    for (b, l, h), u in units.items():
        assert np.sqrt(am.mass_objective(u["E"], u["s"], np.exp(beta[l, h]))) <= RES_TOL * np.linalg.norm(u["s"])


@pytest.mark.parametrize("qdist", ["planted4", "normal", "aligned"])
def test_am_multi_turn_shape_sampled(qdist):
    """The delay-1 multi-turn compaction shape (28 layers, 2 KV heads, 16 query heads x 128 rows:
    R = 2048 > m = 307), 8 sweeps, in the launch configuration the benchmark times; six units
    sampled for the oracle.  With the planted proxy queries token eviction already holds all
    but ~1e-11 of the mass (concentrated units); with diffuse or Q-aligned ones every coordinate
    moves (the aligned recipe is where a coarser rounding guard froze real steps)."""
    import dataclasses
    sp = dataclasses.replace(workloads.spec("multi-turn"), qdist=qdist)
    case = workloads.build(sp, 0, DEV)
    m = [oracle.budget_ratio(n, 0.2) for n in PT.seg_lengths(case)]
    s_orc, _ = oracle.score_cache(case.k_pool, case.block_table, case.nblocks, case.seg_start, case.seg_end,
                                  case.seq_len, case.q, sp.scale)
    keep_np = oracle.select_cache(s_orc, case.seg_start, case.seg_end, m)
    kb, vb, qb = bits(case.k_pool), bits(case.v_pool), bits(case.q)
    beta, vc = run_gpu(case, m, keep_np, 8, None)
    rng = np.random.default_rng(0)
    sample = [(0, int(l), int(h)) for l, h in zip(rng.choice(sp.L, 6, replace=False), rng.integers(0, sp.H, 6))]
    bt = case.block_table.cpu().numpy()
    units = {}
    for (b, l, h) in sample:
        K = am.gather(kb, bt, l, h, b, 0, sp.lengths[0])
        V = am.gather(vb, bt, l, h, b, 0, sp.lengths[0])
        units[(b, l, h)] = am.unit(am.bf16_to_f64(qb[b, l, h]), K, V, keep_np[l, h, :m[0]], sp.scale, 8)
    kinds = check_units(units, m, beta, vc, 8, sample=sample)
    assert kinds["concentrated" if qdist == "planted4" else "well"] == len(sample)


def test_caller_lse_gives_the_same_fit():
    """kvc_am_fit with the LSE kvc_score wrote for the same rows runs no LSE pass of its own and
    gives bit-identical beta, V_C and V pool (the same pass computed the same numbers); the
    proxy rows span two row ranges of the value fit's Gram product and a ragged last key tile."""
    sp = workloads.custom(L=2, H=2, G=4, d=128, P=16, q=24, lengths=(700, 333), shuffle_pages=True,
                          qdist="normal")
    outs = []
    for use_lse in (False, True):
        case = workloads.build(sp, 11, DEV)
        m = [oracle.budget_ratio(n, 0.2) for n in PT.seg_lengths(case)]
        cp = kvc.Compactor(case.k_pool, case.v_pool, case.tags, case.block_table, case.nblocks, case.free_ids,
                           case.free_top, case.seg_start, case.seg_end, case.seq_len, m, sp.R)
        cp.score(case.q, sp.scale, want_lse=True)
        cp.select()
        beta = torch.full((sp.L, sp.H, max(1, cp.Mtot)), float("nan"), device=DEV)
        vc = torch.full((sp.L, sp.H, max(1, cp.Mtot), sp.d), float("nan"), device=DEV)
        cp.am_fit(case.q, sp.scale, 6, beta=beta, vc=vc, lse=cp.lse if use_lse else None)
        torch.cuda.synchronize()
        PT.device_status_clean()
        outs.append((beta.cpu().numpy(), vc.cpu().numpy(), bits(case.v_pool), cp.keep.cpu().numpy()))
    (b0, v0, p0, k0), (b1, v1, p1, k1) = outs
    np.testing.assert_array_equal(k0, k1)
    np.testing.assert_array_equal(b0.view(np.uint32), b1.view(np.uint32))
    np.testing.assert_array_equal(v0.view(np.uint32), v1.view(np.uint32))
    np.testing.assert_array_equal(p0, p1)
