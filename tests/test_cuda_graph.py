"""The library's calls only enqueue work on the given stream (no host
synchronisation, no allocation), so sequences of them can be recorded in a
CUDA graph. Replaying the graph must give bit-identical results to the same
calls made eagerly."""
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from gated_deltanet_linear_02_gb300 import build, ops
    build.build()
    return ops


def test_decode_steps_replay_from_a_cuda_graph(ops):
    B, steps = 4, 6
    lp = I.layer_params(I.seed_of(40)).to(DEV)
    cp = ops.make_params(lp)
    conv0, S0 = I.initial_states(40, B, torch.bfloat16, device=DEV)
    st = I.streams(40, B, torch.bfloat16, device=DEV, lead=(steps,))

    def run(conv, S, outs):
        for k in range(steps):
            ops.decode_step(None, st.qkv[k], st.z[k], st.alpha[k], st.beta[k], conv, S, outs[k], cparams=cp)

    # eager
    conv_e, S_e = conv0.clone(), S0.clone()
    out_e = [torch.empty(B, I.D_INNER, device=DEV) for _ in range(steps)]
    run(conv_e, S_e, out_e)
    # graph: warm up on a side stream, capture, restore the states, replay once
    conv_g, S_g = conv0.clone(), S0.clone()
    out_g = [torch.empty(B, I.D_INNER, device=DEV) for _ in range(steps)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(conv_g, S_g, out_g)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(conv_g, S_g, out_g)
    conv_g.copy_(conv0)
    S_g.copy_(S0)
    graph.replay()
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    for a, b in zip(out_e, out_g):
        assert torch.equal(a, b)
    assert torch.equal(S_e, S_g) and torch.equal(conv_e, conv_g)


def test_attention_and_prefill_replay_from_a_cuda_graph(ops):
    a = I.attn_inputs(41, 3, 700, [700, 129, 1]).to(DEV)
    ws = torch.empty(ops.attn_decode_workspace_size(3, 700), dtype=torch.uint8, device=DEV)
    out_e, out_g = torch.empty(3, 16, 256, device=DEV), torch.empty(3, 16, 256, device=DEV)
    ops.attn_decode(a.q, a.k_cache, a.v_cache, a.ctx_len, a.z, out_e, workspace=ws)
    lp = I.layer_params(I.seed_of(42)).to(DEV)
    cp = ops.make_params(lp)
    lens = [1500, 837]            # longer than one 1024-token window: two window sets on two streams
    st = I.streams(42, sum(lens), torch.bfloat16, device=DEV)
    cu = I.cu_seqlens(lens).to(DEV)
    pws = torch.empty(ops.prefill_workspace_size(2, sum(lens), torch.bfloat16, 0), dtype=torch.uint8, device=DEV)
    pout_e, pout_g = (torch.empty(sum(lens), I.D_INNER, device=DEV) for _ in range(2))
    S_e, S_g = (torch.empty(2, I.HV, I.DV, I.DK, device=DEV) for _ in range(2))
    ops.prefill(None, st.qkv, st.z, st.alpha, st.beta, cu, pout_e, ssm_state_out=S_e, workspace=pws, cparams=cp)

    def body():
        ops.attn_decode(a.q, a.k_cache, a.v_cache, a.ctx_len, a.z, out_g, workspace=ws)
        ops.prefill(None, st.qkv, st.z, st.alpha, st.beta, cu, pout_g, ssm_state_out=S_g, workspace=pws,
                    cparams=cp)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    out_g.zero_()
    pout_g.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ops.device_error() == ops.GDN_OK
    assert torch.equal(out_e, out_g)
    assert torch.equal(pout_e, pout_g) and torch.equal(S_e, S_g)
