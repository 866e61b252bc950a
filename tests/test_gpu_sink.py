"""GPU parity with one dominant key per request over a long row (an
attention sink), against the CPU oracle's exact softmax.

The tensor-core kernel scales the softmax weights to the row's running max
and carries them in e4m3 terms. Keys far below the max are the hard case for
such a representation: here the sink's logit sits about 20 binades (about
14 nats) above n near-equal others, so each other key weighs about 2^-20 of
the sink, and together they hold n * 2^-20 of the weight (1/32 at 32,768
keys, 1/8 at 131,072). A kernel that rounded them to zero would return the
sink's V row; the exact output is a visible mix of the two, which each case
checks first. Rows are compared element by element within the usual
tolerance, unsplit and split (the split partials go through mj_merge_lse),
for both decode kernels.
"""

import numpy as np
import pytest

import synth
from oracle import attention as OA
from tests._harness import all_units, compare, run_gpu, run_oracle, unit_rows, vmax_of

pytestmark = pytest.mark.gpu

IMPLS = [2, 1]  # MJ_IMPL_TCGEN05, MJ_IMPL_SIMT

# name -> (lengths, sink positions (negative: from the end))
CASES = {
    "long_single_131072": ([131072], [0]),
    "four_rows_32768": ([32768, 32768, 32768, 32768], [0, 5000, -1, 20000]),
    # 64/8 heads: 8-row tiles (tile pairs, two P buffers, the single-bound exchange)
    "gqa8_two_rows_32768": ([32768, 32768], [7, -3], dict(h_q=64)),
}
# plans: unsplit, and split the way the long-context benchmark plans
PLANS = {"unsplit": dict(ctas_per_sm=2, max_splits=1), "split": dict(ctas_per_sm=2, max_splits=64)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_fp8_decode_gb300.build import build

    build()


_cache = {}


def _workload(name):
    if name not in _cache:
        lens, pos, *kw = CASES[name]
        w = synth.sink_case(name=name, seq_lens=lens, sink_pos=pos, gap_binades=20.0, **(kw[0] if kw else {}))
        ref, lse, _, _ = run_oracle(w)
        _cache.clear()
        _cache[name] = (w, ref, lse)
    return _cache[name]


@pytest.mark.parametrize("plan", list(PLANS))
@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("impl", IMPLS)
def test_dominant_key_over_a_long_row(impl, name, plan):
    w, ref, lse = _workload(name)
    units = all_units(w)
    # the others' share is visible in the exact output: dropping them (the
    # output = the sink's dequantized V row) would leave the tolerance
    vm = vmax_of(w, units)
    for b, g in units:
        rs, hs = unit_rows(w, b, g)
        _, vc = OA.gather_unit(w.logical("k"), w.logical("v"), w.block_table, b, g, int(w.seq_lens[b]),
                               w.page_size, w.kv_format)
        v_sink = OA.decode_codes(vc[w.meta["sink_pos"][b]], w.kv_format) * OA.descale_at(w.v_scale, b, g)
        assert np.abs(ref[rs, hs] - v_sink).max() > 2e-2 * vm, "the other keys' share must be visible"
    q_mode = "fp8_fused" if plan == "split" else "fp8"
    got = run_gpu(w, impl=impl, q_mode=q_mode, **PLANS[plan])
    assert bool(got["info"]["with_reduction"]) == (plan == "split")
    if plan == "split":
        assert max(got["info"]["n_splits"][: w.num_seqs]) > 1
    compare(w, got["out"], ref, units, f"{name} {plan} impl={impl}")
    np.testing.assert_allclose(got["lse"], lse, atol=2e-3, rtol=1e-4)
    assert got["status"] == 0
