"""Host logic of the step driver that needs no GPU: the buffers a
DataParallelStep sets up for each gathered layout (built here with CPU
tensors and a stand-in stream; nothing is launched)."""
import pytest

import synth
from zero_sharded_optimizer_02_gb300.step import DataParallelStep


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("mode", ["full", "slot", "pitched"])
def test_driver_buffers(mode, fused):
    w = synth.WORKLOADS["c0"]
    psi, nd, bucket = 40_003, 4, 4096
    d = DataParallelStep(psi, nd, range(nd), w.grad_dtype, w.hparams, w.loss_scale, bucket,
                         "cpu", gathered=mode, fused=fused, stream="stand-in")
    s = int(d.layouts[0].shard_elems)
    assert s == 10_001
    assert len(d.gathered) == 2
    for g in d.gathered:
        if mode == "full":
            assert tuple(g.shape) == (nd * s + 8,)
        elif mode == "pitched":
            assert tuple(g.shape) == (nd, int(d.layouts[0].row_pitch))
        else:
            assert sorted(g) == list(range(nd)) and all(t.numel() == s + 8 for t in g.values())
    # the fusion buffer of the unfused path: the bucket (or the shard, if
    # shorter) plus 4 elements for the 16-byte phase shift
    assert d.cb_elems == (0 if fused else min(bucket, s) + 4)
    assert (d.cb is None) == fused


def test_unknown_gathered_layout_is_refused():
    w = synth.WORKLOADS["c0"]
    with pytest.raises(ValueError):
        DataParallelStep(w.psi, w.nd, [0], w.grad_dtype, w.hparams, w.loss_scale, w.bucket,
                         "cpu", gathered="rows", stream="stand-in")
