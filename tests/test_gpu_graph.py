"""The main entry points inside a CUDA graph: after one warm-up call per device (which
does the library's one-time set-up), forward + backward captured into a graph and
replayed give exactly the eager results."""
import pytest
import torch

import workloads
from gpu_util import dev, dev_bf16

pytestmark = pytest.mark.gpu


def test_graph_replay_matches_eager_bitwise():
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as rlk
    w = workloads.Workload("graph", T=300, H=512, V=20480, V_true=20000, seed=51)
    d = workloads.make_inputs(w)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    T, H, V = w.T, w.H, w.V
    logp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    dH = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((V, H), device="cuda")
    fws = torch.empty(rlk.fwd_workspace_bytes(T, H, V), dtype=torch.uint8, device="cuda")
    bws = torch.empty(rlk.bwd_workspace_bytes(T, H, V), dtype=torch.uint8, device="cuda")

    def step():
        rlk.linear_logp_fwd(h, W, y, w.V_true, out=(logp, lse), workspace=fws)
        rlk.linear_logp_bwd(h, W, y, lse, g, w.V_true, out=(dH, dW), workspace=bws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up: one-time per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [x.clone() for x in (logp, lse, dH, dW)]
    for x in (logp, lse, dH, dW):
        x.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (logp, lse, dH, dW)):
        assert torch.equal(a, b)
    # replay with new inputs in the same buffers follows them
    h.copy_(torch.roll(h, 1, dims=0))
    y.copy_(torch.roll(y, 1))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(logp, torch.roll(eager[0], 1))


def test_graph_replay_fp8_path_matches_eager_bitwise():
    """The FP8 step (quantize W and h, FP8 forward, straight-through backward) inside a
    CUDA graph gives the eager bits."""
    from deterministic_token_logprob_gb300 import build
    build.build()
    import deterministic_token_logprob_gb300 as rlk
    w = workloads.Workload("graph8", T=300, H=512, V=20480, V_true=20000, seed=52)
    d = workloads.make_inputs(w)
    h, W, y, g = dev_bf16(d["h"]), dev_bf16(d["W"]), dev(d["y"]), dev(d["g"])
    T, H, V = w.T, w.H, w.V
    hq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    hs = torch.empty(T, device="cuda")
    Wq = torch.empty((V, H), dtype=torch.uint8, device="cuda")
    Ws = torch.empty(V, device="cuda")
    logp = torch.empty(T, device="cuda")
    lse = torch.empty(T, device="cuda")
    dH = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((V, H), device="cuda")
    fws = torch.empty(rlk.fwd_workspace_bytes(T, H, V), dtype=torch.uint8, device="cuda")
    bws = torch.empty(rlk.bwd_workspace_bytes(T, H, V), dtype=torch.uint8, device="cuda")

    def step():
        rlk.quantize_rows_e4m3(W, out=(Wq, Ws))
        rlk.quantize_rows_e4m3(h, out=(hq, hs))
        rlk.linear_logp_fwd_fp8(hq, hs, Wq, Ws, y, w.V_true, out=(logp, lse), workspace=fws)
        rlk.linear_logp_bwd_fp8(h, W, hq, hs, Wq, Ws, y, lse, g, w.V_true, out=(dH, dW),
                                workspace=bws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    outs = (hq, hs, Wq, Ws, logp, lse, dH, dW)
    eager = [x.clone() for x in outs]
    for x in outs:
        x.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
