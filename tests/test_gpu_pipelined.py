"""The pipelined driver (speculative launch of up to `depth` steps before the
oldest one's flag is read) reproduces the plain driver bit for bit,
including a global skip in the middle of the sequence, which forces the
speculative steps to be discarded and run again."""
import dataclasses

import pytest
import torch

import synth
from gpu_util import DEV, TORCH_DT, make_group
from zero_sharded_optimizer_02_gb300.step import PipelinedStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_sharded_optimizer_02_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("depth", [1, 2, 3])
@pytest.mark.parametrize("skip_at", [None, 0, 3, 5])
def test_pipelined_equals_plain(skip_at, depth):
    w = dataclasses.replace(synth.WORKLOADS["c0"], psi=300_007, nd=8, plant=None,
                            fresh_grads=True)
    steps = 6
    plain = make_group(w, gathered="full", bucket=40_000)
    pipe = PipelinedStep(w.psi, w.nd, range(w.nd), w.grad_dtype, w.hparams, w.loss_scale,
                         40_000, DEV, gathered="full", depth=depth)
    for r in range(w.nd):
        pipe.state[r].bufs[0].copy_(plain.state[r].bufs[plain.state[r].cur])
    pitch = int(plain.layouts[0].row_pitch)
    s = int(plain.layouts[0].shard_elems)
    bufs = []
    for k in range(steps):                       # every step keeps its own gradients
        b = torch.empty(w.nd, w.nd * pitch, dtype=TORCH_DT[w.grad_dtype], device=DEV)
        synth.fill_full_rows(w, k, b)
        if k == skip_at:
            b[3, 2 * pitch + s // 3] = float("inf")
        bufs.append(b)
    import zero_sharded_optimizer_02_gb300 as z
    descs = [{r: z.grads(b, w.nd * pitch, r * pitch, w.nd, w.grad_dtype) for r in range(w.nd)}
             for b in bufs]
    expect = [plain.step(d) for d in descs]
    got = []
    for d in descs:
        got += pipe.launch(d)
    got += pipe.finish()
    assert got == expect == [k == skip_at for k in range(steps)]
    assert pipe.t == plain.t
    for r in range(w.nd):
        for a, b in zip(pipe.state[r].tensors(), plain.state[r].tensors()):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(pipe.gathered_view()[:w.psi].view(torch.int16),
                       plain.gathered_view()[:w.psi].view(torch.int16))
    assert not pipe.flags.any()
