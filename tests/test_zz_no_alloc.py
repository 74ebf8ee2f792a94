"""The allocation-free top-k entry point, ts_topk_noalloc.

Some callers cannot call cudaMalloc: a plugin running inside a host engine
that owns every device allocation, or a process whose device memory was all
reserved before it started. For them the library offers a top-k whose scratch
is a fixed device array inside the library. This test calls it through the C
ABI and checks it against ts_topk with a caller workspace, and a few requests
against the CPU oracle, on calls in a row: the one-launch path, then the
long-context path twice with different shapes (that path's histograms and
counters live in the shared array, so the second call must clear what the
first left there). It also checks that sizes past its limit are refused up
front. It sits in a file of its own that pytest collects last."""
import numpy as np
import pytest

from _util import ensure_library

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import decode_dsa_kv_gb300 as d
    return d


def _inputs(rng, B, ctx, ties):
    s = rng.standard_normal((B, ctx)).astype(np.float32)
    if ties:
        s = np.round(s * 2) / 2            # few distinct values: many exact ties
    return s


def test_noalloc_matches_workspace_topk_on_calls_in_a_row(d):
    import oracle
    rng = np.random.default_rng(2024)
    # one-launch path, then the long-context path at the limit (2 x 2^21) and
    # again at another shape (4 x 2^20)
    cases = [(32, 65536, 2048, False), (2, 1 << 21, 2048, True), (4, 1 << 20, 2048, True)]
    for B, ctx, k, ties in cases:
        scores = torch.from_numpy(_inputs(rng, B, ctx, ties)).cuda()
        lens = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = torch.empty((B, k), dtype=torch.int32, device="cuda")
        nbytes = d.ts_topk_workspace_size(B, ctx, k)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        assert d.ts_topk(scores, ctx, lens, B, ctx, k, ref, ws, nbytes, err) == 0
        got = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        assert d.ts_topk_noalloc(scores, ctx, lens, B, ctx, k, got, err) == 0
        assert d.ts_read_error(err) == 0
        assert torch.equal(got, ref), (B, ctx, k)
        host_scores = scores.cpu().numpy()
        for b in (0, B - 1):
            assert np.array_equal(got[b].cpu().numpy(), oracle.topk_ids(host_scores[b], ctx, k)), \
                (B, ctx, b)


def test_noalloc_refuses_sizes_past_its_limit(d):
    from decode_dsa_kv_gb300 import _abi
    scores = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    lens = torch.full((1,), 64, dtype=torch.int32, device="cuda")
    ids = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    # more requests than the scratch holds, and more positions than it holds;
    # both refused on the host before anything is enqueued
    assert d.ts_topk_noalloc(scores, 64, lens, 129, 64, 8, ids) == _abi.TS_ERR_UNSUPPORTED
    assert d.ts_topk_noalloc(scores, 1 << 22, lens, 2, (1 << 21) + 1, 8, ids) == \
        _abi.TS_ERR_UNSUPPORTED
