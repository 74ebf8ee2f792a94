"""Per-kernel parity of the CUDA path (through the C ABI) with the CPU oracle:
bit-exact for top-k, plan, gather and refill; within the stated tolerance for
SFA. Plus the device-side error reporting of bad data."""
import math

import numpy as np
import pytest

import oracle
import workload as wl
from _util import SFA_ABS_TOL, SFA_MEAN_REL_TOL, ensure_library, sfa_errors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import decode_dsa_kv_gb300 as d
    return d


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------

def run_topk(d, scores: np.ndarray, lens: np.ndarray, k: int, max_ctx=None):
    B, stride = scores.shape
    max_ctx = int(lens.max()) if max_ctx is None else max_ctx
    s = torch.from_numpy(scores).cuda()
    ln = torch.from_numpy(lens.astype(np.int32)).cuda()
    ids = torch.empty((B, k), dtype=torch.int32, device="cuda")
    nbytes = d.ts_topk_workspace_size(B, max_ctx, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = _err()
    assert d.ts_topk(s, stride, ln, B, max_ctx, k, ids, ws, nbytes, err) == 0
    bits = d.ts_read_error(err)
    return ids.cpu().numpy(), bits


def _check_topk(d, scores, lens, k):
    ids, bits = run_topk(d, scores, lens, k)
    assert bits == 0
    for b in range(scores.shape[0]):
        want = oracle.topk_ids(scores[b], int(lens[b]), k)
        assert np.array_equal(ids[b], want), f"request {b}"


def test_topk_small_ragged_with_ties(d):
    rng = np.random.default_rng(1)
    lens = np.array([100, 257, 4096, 64], np.int32)
    scores = np.full((4, 4096), np.nan, np.float32)
    for b, n in enumerate(lens):
        scores[b, :n] = np.round(rng.standard_normal(n) * 3) / 3
    scores[1, :10] = -0.0
    scores[1, 10:20] = 0.0
    scores[2, 5] = np.inf
    scores[2, 6] = -np.inf
    for k in (1, 7, 64):
        _check_topk(d, scores, lens, k)


def test_topk_all_equal_and_k_equals_ctx(d):
    scores = np.full((2, 20000), 1.5, np.float32)
    lens = np.array([20000, 2048], np.int32)
    _check_topk(d, scores, lens, 2048)
    scores2 = np.random.default_rng(2).standard_normal((1, 3000)).astype(np.float32)
    _check_topk(d, scores2, np.array([3000], np.int32), 3000)
    # many requests (one CTA each): every score tied in some of them, so the
    # candidate list outgrows shared memory
    rng = np.random.default_rng(3)
    scores4 = np.round(rng.standard_normal((96, 10000)) * 2).astype(np.float32)
    scores4[::7] = 0.5
    _check_topk(d, scores4, np.full(96, 10000, np.int32), 2048)
    # past the one-CTA-per-request size: the many-CTA path, every score tied
    scores3 = np.full((2, 150016), -2.25, np.float32)
    _check_topk(d, scores3, np.array([150016, 140001], np.int32), 2048)


def test_topk_errors(d):
    scores = np.zeros((2, 64), np.float32)
    scores[0, 3] = np.nan
    lens = np.array([64, 10], np.int32)
    ids, bits = run_topk(d, scores, lens, 16, max_ctx=64)
    assert bits & 0x02                          # NaN in request 0
    assert bits & 0x10                          # request 1: ctx 10 < k 16
    assert np.all(ids[1] == -1)


@pytest.mark.parametrize("name", ["tiny", "decode_batch", "long_context", "large_batch",
                                  "adversarial"])
def test_topk_workloads_full_size(d, name):
    w = wl.get(name)
    stream = wl.ScoreStream(w)
    lens = wl.ctx_lens(w)
    for _ in range(2 if name in ("tiny", "adversarial") else 1):
        _check_topk(d, stream.next(), lens, w.k)


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def _random_state(rng, B, S, W, ctx, fill=0.7):
    tags = np.full((B, S * W), -1, np.int32)
    ptr = rng.integers(0, W, size=(B, S)).astype(np.int32)
    for b in range(B):
        for s in range(S):
            cands = np.arange(s, ctx, S)
            n = min(len(cands), int(rng.binomial(W, fill)))
            if n:
                tags[b, s * W: s * W + n] = rng.choice(cands, n, replace=False)
    return tags, ptr


def run_plan(d, ids, lens, tags, ptr, S, W):
    B, k = ids.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    i32 = lambda *s: torch.full(s, -7, dtype=torch.int32, device="cuda")
    out = dict(src_map=i32(B, k), miss_ids=i32(B, k), miss_pos=i32(B, k), victim=i32(B, k),
               install=torch.zeros((B, k), dtype=torch.uint8, device="cuda"),
               miss_count=i32(B), miss_rows=i32(B), ptr_next=i32(B, S))
    err = _err()
    st = d.dsa_plan(t(ids), t(lens), B, k, t(tags), t(ptr), S, W, out["src_map"],
                    out["miss_ids"], out["miss_pos"], out["victim"], out["install"],
                    out["miss_count"], out["miss_rows"], out["ptr_next"], err)
    assert st == 0
    bits = d.ts_read_error(err)
    return {n: v.cpu().numpy() for n, v in out.items()}, bits


def _check_plan(d, ids, lens, tags, ptr, S, W):
    got, bits = run_plan(d, ids, lens, tags, ptr, S, W)
    assert bits == 0
    for b in range(ids.shape[0]):
        want = oracle.dsa_plan(ids[b], int(lens[b]), tags[b], ptr[b], S, W)
        M = want.miss_count
        assert got["miss_count"][b] == M
        assert got["miss_rows"][b] == want.miss_rows
        assert np.array_equal(got["src_map"][b], want.src_map)
        assert np.array_equal(got["miss_ids"][b, :M], want.miss_ids)
        assert np.array_equal(got["miss_pos"][b, :M], want.miss_pos)
        assert np.array_equal(got["victim"][b, :M], want.victim)
        assert np.array_equal(got["install"][b, :M], want.install_code)
        assert np.array_equal(got["ptr_next"][b], want.ptr_next)
    return got


@pytest.mark.parametrize("S,W,k,ctx", [(256, 4, 256, 4096), (512, 16, 2048, 65536),
                                       (1024, 16, 2048, 200000), (2, 2, 64, 64),
                                       (37, 3, 100, 1000)])
def test_plan_random_sorted(d, S, W, k, ctx):
    rng = np.random.default_rng(S + W + k)
    B = 5
    tags, ptr = _random_state(rng, B, S, W, ctx)
    lens = np.full(B, ctx, np.int32)
    ids = np.stack([np.sort(rng.choice(ctx, k, replace=False)) for _ in range(B)]).astype(np.int32)
    # request 0 keeps many of its tagged tokens (hits), request 1 floods one set
    held = tags[0][tags[0] >= 0]
    take = min(k // 2, held.size)
    ids[0] = np.sort(np.concatenate([rng.choice(held, take, replace=False),
                                     rng.choice(np.setdiff1d(np.arange(ctx), held), k - take,
                                                replace=False)]))
    flood = np.arange(3 % S, ctx, S)[: min(k // 2, 3 * W + 5)]
    rest = rng.choice(np.setdiff1d(np.arange(ctx), flood), k - flood.size, replace=False)
    ids[1] = np.sort(np.concatenate([flood, rest]))
    _check_plan(d, ids, lens, tags, ptr, S, W)


def test_plan_unsorted_with_repeats(d):
    rng = np.random.default_rng(9)
    S, W, k, ctx, B = 64, 4, 512, 5000, 3
    tags, ptr = _random_state(rng, B, S, W, ctx)
    lens = np.full(B, ctx, np.int32)
    ids = rng.integers(0, 700, size=(B, k)).astype(np.int32)
    _check_plan(d, ids, lens, tags, ptr, S, W)


def test_plan_bad_ids_flagged(d):
    S, W, k = 8, 2, 16
    tags = np.full((1, S * W), -1, np.int32)
    ptr = np.zeros((1, S), np.int32)
    ids = np.arange(k, dtype=np.int32)[None].copy()
    ids[0, 5] = 99                      # past ctx_len 50
    got, bits = run_plan(d, ids, np.array([50], np.int32), tags, ptr, S, W)
    assert bits & 0x01
    assert got["src_map"][0, 5] == np.iinfo(np.int32).min
    assert got["miss_count"][0] == k - 1


# ---------------------------------------------------------------------------
# gather and refill
# ---------------------------------------------------------------------------

def test_gather_and_refill_bytes(d):
    from decode_dsa_kv_gb300 import HostKV
    rng = np.random.default_rng(4)
    B, S, W, k, ctx = 3, 64, 4, 300, 3000
    P = S * W
    host = HostKV(1, B, ctx)
    host.array[...] = rng.integers(0, 65536, size=host.array.shape, dtype=np.uint16)
    pool = rng.integers(0, 65536, size=(B, P, 576), dtype=np.uint16)
    tags, ptr = _random_state(rng, B, S, W, ctx)
    lens = np.array([ctx, 2000, 1500], np.int32)
    ids = np.stack([np.sort(rng.choice(int(n), k, replace=False)) for n in lens]).astype(np.int32)
    for b in range(B):                     # make the pool hold the tagged rows
        for slot in np.flatnonzero(tags[b] >= 0):
            pool[b, slot] = host.array[0, b, tags[b, slot]]
    got, bits = run_plan(d, ids, lens, tags, ptr, S, W)
    assert bits == 0
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pool_t = t(pool.view(np.int16))
    sel = torch.zeros((B, k, 576), dtype=torch.int16, device="cuda")
    err = _err()
    ln = t(lens)
    assert d.dsa_gather_kv(t(got["src_map"]), t(got["miss_ids"]), t(got["miss_pos"]),
                           t(got["miss_count"]), t(got["miss_rows"]), B, k, pool_t, P,
                           host.layer_ptr(0), ctx, ln, sel, err) == 0
    assert d.ts_read_error(err) == 0
    sel_np = sel.cpu().numpy().view(np.uint16)
    for b in range(B):
        want = oracle.dsa_serve(got["src_map"][b], pool[b], host.array[0, b], int(lens[b]))
        assert np.array_equal(sel_np[b], want)
        assert np.array_equal(sel_np[b], host.array[0, b][ids[b]])
    # refill with metadata update
    tags_t, ptr_t = t(tags), t(ptr)
    assert d.dsa_refill_pool(t(got["miss_ids"]), t(got["miss_pos"]), t(got["victim"]),
                             t(got["install"]), t(got["miss_count"]), B, k, sel, pool_t, P, 1,
                             tags_t, ptr_t, t(got["ptr_next"]), S, W, err) == 0
    assert d.ts_read_error(err) == 0
    pool_after = pool_t.cpu().numpy().view(np.uint16)
    for b in range(B):
        plan = oracle.dsa_plan(ids[b], int(lens[b]), tags[b], ptr[b], S, W)
        pb = pool[b].copy()
        oracle.dsa_install(pb, plan, host.array[0, b])
        tb, qb = tags[b].copy(), ptr[b].copy()
        oracle.metadata_update(tb, qb, plan)
        assert np.array_equal(pool_after[b], pb)
        assert np.array_equal(tags_t[b].cpu().numpy(), tb)
        assert np.array_equal(ptr_t[b].cpu().numpy(), qb)
    host.close()


def test_gather_flags_bad_rows(d):
    from decode_dsa_kv_gb300 import HostKV
    host = HostKV(1, 1, 64)
    pool = torch.zeros((1, 8, 576), dtype=torch.int16, device="cuda")
    sel = torch.zeros((1, 4, 576), dtype=torch.int16, device="cuda")
    src = torch.tensor([[0, 9, -1 - 70, -1 - 3]], dtype=torch.int32, device="cuda")
    mids = torch.tensor([[3, 70, 0, 0]], dtype=torch.int32, device="cuda")
    mpos = torch.tensor([[3, 2, 0, 0]], dtype=torch.int32, device="cuda")
    mcnt = torch.tensor([2], dtype=torch.int32, device="cuda")
    err = _err()
    ln = torch.tensor([64], dtype=torch.int32, device="cuda")
    assert d.dsa_gather_kv(src, mids, mpos, mcnt, mcnt, 1, 4, pool, 8, host.layer_ptr(0), 64, ln,
                           sel, err) == 0
    bits = d.ts_read_error(err)
    assert bits & 0x04 and bits & 0x01
    host.close()


def test_gather_repeated_ids(d):
    """Caller-supplied ids with repeats: every copy of a missed token gets its
    host row (the miss list serves the first position, the second pass the
    others)."""
    from decode_dsa_kv_gb300 import HostKV
    rng = np.random.default_rng(8)
    S, W, k, ctx = 16, 2, 200, 300
    host = HostKV(1, 1, ctx)
    host.array[...] = rng.integers(0, 65536, size=host.array.shape, dtype=np.uint16)
    tags, ptr = _random_state(rng, 1, S, W, ctx)
    pool = np.zeros((1, S * W, 576), np.uint16)
    for slot in np.flatnonzero(tags[0] >= 0):
        pool[0, slot] = host.array[0, 0, tags[0, slot]]
    ids = rng.integers(0, 120, size=(1, k)).astype(np.int32)
    lens = np.array([ctx], np.int32)
    got, bits = run_plan(d, ids, lens, tags, ptr, S, W)
    assert bits == 0
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    sel = torch.zeros((1, k, 576), dtype=torch.int16, device="cuda")
    err = _err()
    assert got["miss_rows"][0] > got["miss_count"][0]      # the ids do repeat
    assert d.dsa_gather_kv(t(got["src_map"]), t(got["miss_ids"]), t(got["miss_pos"]),
                           t(got["miss_count"]), t(got["miss_rows"]), 1, k,
                           t(pool.view(np.int16)), S * W, host.layer_ptr(0), ctx, t(lens), sel,
                           err) == 0
    assert d.ts_read_error(err) == 0
    assert np.array_equal(sel.cpu().numpy().view(np.uint16)[0], host.array[0, 0][ids[0]])
    host.close()


# ---------------------------------------------------------------------------
# SFA
# ---------------------------------------------------------------------------

def run_sfa(d, q_bits, rows_bits, scale):
    B, H, _ = q_bits.shape
    k = rows_bits.shape[1]
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    sel = torch.from_numpy(rows_bits.view(np.int16)).cuda()
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    nbytes = d.sfa_workspace_size(B, H, k)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    err = _err()
    assert d.sfa_mla_decode(q, sel, B, H, k, scale, out, lse, ws, nbytes, err) == 0
    assert d.ts_read_error(err) == 0
    return out.cpu().view(torch.int16).numpy().view(np.uint16), lse.cpu().numpy()


@pytest.mark.parametrize("B,H,k", [(1, 16, 256), (2, 128, 2048), (3, 128, 300), (1, 128, 1),
                                   (2, 20, 513), (1, 256, 1000), (4, 128, 4096), (2, 128, 1800),
                                   (1, 512, 2048),
                                   (3, 64, 1279)])
def test_sfa_parity(d, B, H, k):
    rng = np.random.default_rng(B * 1000 + H + k)
    q = wl.normal_bf16(B * H, 576, 77, 9, B, H).reshape(B, H, 576)
    rows = wl.normal_bf16(B * k, 576, 78, 9, B, k).reshape(B, k, 576)
    scale = 1 / math.sqrt(576)
    out, lse = run_sfa(d, q, rows, scale)
    worst_abs, rels = 0.0, []
    for b in range(B):
        o, z = oracle.sfa_decode(q[b], rows[b], scale)
        a, r = sfa_errors(out[b], oracle.round_to_bf16_bits(o))
        worst_abs = max(worst_abs, a)
        rels.append(r)
        assert np.allclose(lse[b], z, rtol=0, atol=2e-3)
    assert worst_abs <= SFA_ABS_TOL, worst_abs
    assert max(rels) <= SFA_MEAN_REL_TOL, rels


@pytest.mark.parametrize("next_n", [1, 2, 3])
def test_sfa_mtp_folded_queries_match_separate_calls(d, next_n):
    """MTP reuse (GLM-5.2 shared-Indexer KV Cache Offload, §5.1): the draft
    steps reuse the first step's selection, and their queries are folded into
    the attention's head dimension, (1 + next_n) x 128 heads in one call. Each
    head tile is computed on its own, so the folded call equals one call per
    draft step bit for bit."""
    B, H, k = 3, 128, 2048
    Hf = (1 + next_n) * H
    q = wl.normal_bf16(B * Hf, 576, 81, 9, next_n, 0).reshape(B, Hf, 576)
    rows = wl.normal_bf16(B * k, 576, 82, 9, next_n, 0).reshape(B, k, 576)
    scale = 1 / math.sqrt(576)
    out_f, lse_f = run_sfa(d, q, rows, scale)
    for i in range(1 + next_n):
        out_i, lse_i = run_sfa(d, np.ascontiguousarray(q[:, i * H:(i + 1) * H]), rows, scale)
        assert np.array_equal(out_f[:, i * H:(i + 1) * H], out_i)
        assert np.array_equal(lse_f[:, i * H:(i + 1) * H], lse_i)


def test_sfa_constant_rows_exact(d):
    rng = np.random.default_rng(5)
    row = wl.normal_bf16(1, 576, 5, 9, 0, 0)
    rows = np.repeat(row[None], 2048, axis=1).reshape(1, 2048, 576)
    q = wl.normal_bf16(128, 576, 6, 9, 0, 0).reshape(1, 128, 576)
    out, lse = run_sfa(d, q, rows, 1 / 24)
    assert np.array_equal(out[0], np.repeat(row[:, :512], 128, axis=0))


def test_ts_copy_between_device_and_registered_host(d):
    from decode_dsa_kv_gb300 import PinnedHost
    rng = np.random.default_rng(12)
    n = 3 * 1024 * 1024 + 48
    h_in = PinnedHost((n,), np.uint8)
    h_in.array[:] = rng.integers(0, 256, n, dtype=np.uint8)
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")
    h_out = PinnedHost((n,), np.uint8)
    assert d.ts_copy(dev, h_in.dev, n) == 0            # host -> device
    assert d.ts_copy(h_out.dev, dev, n) == 0           # device -> host
    torch.cuda.synchronize()
    assert np.array_equal(dev.cpu().numpy(), h_in.array)
    assert np.array_equal(h_out.array, h_in.array)
    assert d.ts_copy(dev, h_in.dev, 15) != 0           # not a multiple of 16 bytes
    h_in.close()
    h_out.close()


# ---------------------------------------------------------------------------
# adjacent-step reuse plan
# ---------------------------------------------------------------------------

def _plan_reuse(d, ids, prev, lens):
    B, k = ids.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    out = {n: torch.zeros((B, k), dtype=torch.int32, device="cuda")
           for n in ("src_map", "miss_ids", "miss_pos")}
    mc = torch.zeros(B, dtype=torch.int32, device="cuda")
    mr = torch.zeros(B, dtype=torch.int32, device="cuda")
    err = _err()
    assert d.dsa_plan_reuse(t(ids), t(prev), t(lens), B, k, out["src_map"], out["miss_ids"],
                            out["miss_pos"], mc, mr, err) == 0
    bits = d.ts_read_error(err)
    return {n: v.cpu().numpy() for n, v in out.items()}, mc.cpu().numpy(), mr.cpu().numpy(), bits


@pytest.mark.parametrize("B,k,ctx,overlap", [(3, 300, 3000, 0.6), (2, 2048, 65536, 0.6),
                                             (1, 1, 10, 1.0), (2, 513, 100000, 0.0)])
def test_plan_reuse_matches_oracle(d, B, k, ctx, overlap):
    rng = np.random.default_rng(k + B)
    prev = np.stack([np.sort(rng.choice(ctx, k, replace=False)) for _ in range(B)]).astype(np.int32)
    ids = []
    for b in range(B):
        keep = rng.choice(prev[b], int(round(overlap * k)), replace=False)
        rest = rng.choice(np.setdiff1d(np.arange(ctx), prev[b]), k - keep.size, replace=False)
        ids.append(np.sort(np.concatenate([keep, rest])))
    ids = np.stack(ids).astype(np.int32)
    lens = np.full(B, ctx, np.int32)
    got, mc, mr, bits = _plan_reuse(d, ids, prev, lens)
    assert bits == 0
    for b in range(B):
        p = oracle.plan_reuse(ids[b], prev[b], ctx)
        assert np.array_equal(got["src_map"][b], p.src_map)
        assert mc[b] == p.miss_count and mr[b] == p.miss_rows
        assert np.array_equal(got["miss_ids"][b, :mc[b]], p.miss_ids)
        assert np.array_equal(got["miss_pos"][b, :mc[b]], p.miss_pos)


def test_plan_reuse_first_step_and_bad_input(d):
    ids = np.array([[2, 5, 9]], np.int32)
    got, mc, _, bits = _plan_reuse(d, ids, np.full((1, 3), -1, np.int32), np.array([10], np.int32))
    assert bits == 0 and mc[0] == 3 and got["src_map"][0].tolist() == [-3, -6, -10]
    _, _, _, bits = _plan_reuse(d, np.array([[2, 12, 9]], np.int32), np.full((1, 3), -1, np.int32),
                                np.array([10], np.int32))
    from decode_dsa_kv_gb300 import _abi
    assert bits & _abi.TS_DEVERR_ID_RANGE      # 12 is past the context
    assert bits & _abi.TS_DEVERR_ORDER         # 12 then 9: not ascending
