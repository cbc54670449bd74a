"""The library's launches can be captured in a CUDA graph and replayed: kda_fwd (both forward
kernels), kda_fwd_ws (the cluster launch of the shared-preparation kernel, workspace allocated
before the capture) and kda_decode, after one eager call on the device (the first call configures
each kernel's shared-memory size and queries the device, host work that is not part of a
capture). Replays must equal eager calls bit for bit."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,shared", [pytest.param(3, False, id="mma"), pytest.param(80, False, id="tcgen05"),
                                      pytest.param(3, True, id="shared-preparation")])
def test_forward_pass_replays_from_a_cuda_graph(H, shared):
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", T=77, H=H, B=1)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    fin = torch.empty_like(c["initial_state"])
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin)
    if shared:
        ws = torch.empty(kda.workspace_bytes(1, H), dtype=torch.uint8, device="cuda")
        assert ws.numel() > 0
        call = lambda: kda.fwd_ws(*args, workspace=ws)
    else:
        call = lambda: kda.fwd(*args)
    call()
    torch.cuda.synchronize()
    kda.check_device_status()
    ref_out, ref_fin = out.clone(), fin.clone()
    out.zero_()
    fin.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    kda.check_device_status()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_decode_steps_replay_from_a_cuda_graph():
    import gated_linear_attention_kda_gb300 as kda
    S, H = 4, 8
    d = W.make("b2_t128_h8", B=S, T=1, H=H)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}  # [S, 1, H, 128] tokens
    state0 = c["initial_state"].clone()
    out = torch.empty_like(c["v"])
    state = state0.clone()
    step = lambda: kda.decode(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, state, c["A_log"],
                              c["dt_bias"], d["lower_bound"])
    for _ in range(3):  # eager: three steps from state0
        step()
    torch.cuda.synchronize()
    kda.check_device_status()
    ref_out, ref_state = out.clone(), state.clone()
    state.copy_(state0)
    out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    state.copy_(state0)  # the capture does not run the step
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    kda.check_device_status()
    assert torch.equal(out, ref_out) and torch.equal(state, ref_state)
