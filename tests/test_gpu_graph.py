"""The owner step replayed from a CUDA graph equals the step issued call by call (bit for bit:
the same kernels on the same inputs), over three steps of the GPT-2-small owned set."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_eager_steps():
    import bench
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    a = bench.Workload(1, 0, dev)
    b = bench.Workload(1, 0, dev)
    hp = a.wl.hyper
    g = b.runner.capture(b.contrib, hp)
    for _ in range(3):
        a.runner.step(a.contrib, a.tail_contrib, hp)
        b.runner.graph_step(g, b.tail_contrib, hp)
    torch.cuda.synchronize()
    for name in ("weights", "momentum", "ortho", "norm", "tail_p", "tail_m", "tail_v"):
        assert torch.equal(getattr(a.runner, name), getattr(b.runner, name)), name
    from matrix_optimizer_owner_gb300 import mfsdp
    assert mfsdp.mfsdp_query_status() == 0
