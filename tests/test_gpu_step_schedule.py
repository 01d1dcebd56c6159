"""bench.py's step graphs for a workload with importance scores: the score update on a second
stream (each layer's logits and LSE in a ring of three buffers) and the score update fused
into each layer's merge launch give the same scores, and both match the oracle's
(1/(L·H)) Σ_t Σ_ℓ Σ_h α sum ([TIER] "2. 중요도 점수화") over all layers and steps."""

import numpy as np
import pytest
import torch

import bench
import harness as H
from kvd_inputs import Workload


def _workload():
    w = Workload("sched", L=3, n_q=8, n_kv=2, d_h=128, batch=2, kv_dtype="bf16", seed=5, steps=3,
                 evict_frac=0.05, protect_prompt=32, protect_recent=16, scores=True)
    w._ctx0 = [600, 333]
    return w


def _run(w, dev, fused):
    st = bench.Step(w, dev, fused_scores=fused)
    graphs = st.capture()   # also runs step 0 once eagerly: start the scores from zero again
    st.scores.zero_()
    for t in range(w.steps):
        graphs[t].replay()
    torch.cuda.synchronize()
    assert st.kvd.kvd_get_device_error(st.pool.handle) == 0
    return st.scores.double().cpu().numpy(), st.out.float().cpu().numpy(), st.bt.cpu()


@pytest.mark.gpu
def test_score_update_on_second_stream_matches_fused_and_oracle(cuda_device):
    w = _workload()
    s_side, out_side, bt = _run(w, cuda_device, fused=False)
    s_fused, out_fused, _ = _run(w, cuda_device, fused=True)
    # same per-layer updates in the same layer order; only the LSE they use is reduced in a
    # different order (merge kernel vs the fused epilogue's own reduction)
    np.testing.assert_allclose(s_side, s_fused, rtol=1e-5, atol=1e-9)
    np.testing.assert_allclose(out_side, out_fused, rtol=1e-2, atol=2e-3)
    retain = w.retain_mask(bt)
    want = np.zeros_like(s_side)
    for t in range(w.steps):
        lens = w.seq_lens(t)
        for layer in range(w.L):
            ref = H.oracle_layer(w, layer, bt, lens, retain=retain, step=t, want_alpha=True)
            for b, n in enumerate(lens):
                want[b, :n] += ref["alpha"][b, :, :n].sum(0) / (w.L * w.n_q)
    assert np.all(np.abs(s_side - want) <= H.SCORE_RTOL * np.abs(want) + 1e-12)
