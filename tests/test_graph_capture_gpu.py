"""Decode steps (kda_recurrent_step) captured in a CUDA graph and replayed give the
same outputs and state as the same calls made one by one: the entry point does
nothing on the host that stream capture forbids, and replays it bit for bit."""
import pytest
import torch

import kda_inputs as ki

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_gb300 as m
    m.build()
    m.load_library()
    return m


def test_decode_steps_replay_from_a_cuda_graph(kda):
    N, H, d, steps = 8, 4, 128, 6
    dev = torch.device("cuda")
    S0 = ki.decode_state(N, H, d, d, seed=31).to(dev)
    ins = [{k: (v.to(dev) if torch.is_tensor(v) else v)
            for k, v in ki.decode_inputs(N, H, d, d, "bf16", seed=31, step=s).items()} for s in range(steps)]
    outs = [torch.empty(N, H, d, dtype=torch.bfloat16, device=dev) for _ in range(steps)]

    def run(S, s):
        for x, o in zip(ins, outs):
            kda.kda_recurrent_step(S, x["q"], x["k"], x["v"], x["g"], x["beta"], scale=x["scale"], out=o, stream=s)

    S_eager = S0.clone()
    run(S_eager, torch.cuda.current_stream())
    o_eager = [o.clone() for o in outs]
    torch.cuda.synchronize()

    S_graph = S0.clone()
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        run(S_graph, cap)
    for o in outs:
        o.zero_()
    torch.cuda.synchronize()
    assert torch.equal(S_graph, S0)  # capture enqueues nothing
    g.replay()
    torch.cuda.synchronize()
    kda.kda_get_device_error()
    assert torch.equal(S_graph, S_eager)
    for a, b in zip(outs, o_eager):
        assert torch.equal(a, b)
