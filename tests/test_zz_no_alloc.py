"""The allocation-free router entry point (for callers that cannot allocate device
memory, e.g. during stream capture or inside an engine that owns the whole device
pool).  Its results must equal the router inside sgp_layer_temporal on the same
residual stream h, on two calls in a row (the calls share one fixed scratch array)."""
import pytest
import torch

from intra_spatial_pipelining_gb300 import sgp, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def test_noalloc_router_matches_the_layer_router_on_two_calls():
    wl = synth.WORKLOADS["gptoss_layer"]
    inp = H.make_inputs(wl, 21)
    d = H.dims(wl.shape)
    ref = H.run_temporal_layer(inp, d)          # the existing entry point, with dumps
    assert ref["status"] == sgp.SGP_OK
    T, k = wl.n_tokens, wl.shape.top_k
    w = inp.weights[0]
    h = ref["dump"]["h"]
    for _ in range(2):
        u = torch.full_like(h, float("nan"))
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        tw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        sgp.sgp_router_topk_noalloc(d, h, w["g_mlp"], w["w_router"], w["router_bias"], T, u,
                                    idx, tw)
        torch.cuda.synchronize()
        H.assert_close("u", u, ref["dump"]["u"].double().cpu().numpy())
        assert torch.equal(idx, ref["idx"])
        assert float((tw - ref["w"]).abs().max()) <= 1e-6


def test_noalloc_router_refuses_sizes_beyond_its_scratch():
    wl = synth.WORKLOADS["gptoss_layer"]
    d = H.dims(wl.shape)
    d.n_experts = 1024                          # 256 tokens x 1024 experts fit ...
    h = torch.zeros(257, wl.shape.hidden, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(wl.shape.hidden, dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros(1024, wl.shape.hidden, dtype=torch.bfloat16, device="cuda")
    u = torch.empty_like(h)
    idx = torch.empty(257, wl.shape.top_k, dtype=torch.int32, device="cuda")
    tw = torch.empty(257, wl.shape.top_k, dtype=torch.float32, device="cuda")
    with pytest.raises(sgp.SgpError) as e:     # ... 257 do not
        sgp.sgp_router_topk_noalloc(d, h, g, wr, None, 257, u, idx, tw)
    assert e.value.code == sgp.SGP_ERR_INVALID_ARG
