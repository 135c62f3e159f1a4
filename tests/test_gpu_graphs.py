"""CUDA-graph capture ("CSA Fused Compressor", section CUDA graphs: warm up each
configuration, pass a static capacity): forward and backward captured once on a
stream and replayed give the eager results bit for bit, for every kernel family
(ratio 4 pipelined and register-window, ratio 128 both window forms, generic ratios)."""
import numpy as np
import pytest

import csa_workloads as w
from gpu_util import Dev, bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ratio,coff,head_dim,lens", [(4, 2, 512, [4096, 37, 3]), (4, 2, 64, [300, 9]),
                                                      (128, 1, 512, [4096, 300]), (128, 2, 128, [1000]),
                                                      (16, 2, 512, [900, 17]), (7, 1, 64, [300, 5]),
                                                      (3, 2, 256, [700, 5])])
def test_capture_and_replay_bitwise(ratio, coff, head_dim, lens):
    import torch
    import sparse_attention_kv_csa_gb300 as csa
    c = w.make_case("graph", ratio, coff, head_dim, lens, extra_rows=2, seed=3)
    d = Dev(c)
    C = coff * head_dim
    out = torch.empty((c.capacity, head_dim), dtype=torch.int16, device="cuda")
    dkv = torch.empty((c.n_tokens, C), dtype=torch.int16, device="cuda")
    dsc = torch.empty_like(dkv)
    dape = torch.empty((ratio, C), dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()

    def step():
        csa.csa_compress_fwd(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, ratio, coff, head_dim, c.capacity, out, st)
        csa.csa_compress_bwd(d.kv, d.score, d.ape, d.cu, d.cc, c.n_seg, ratio, coff, head_dim, c.capacity,
                             c.n_tokens, d.g, dkv, dsc, dape, st)

    with torch.cuda.stream(st):
        step()  # warm-up: per-device set-up happens outside the capture
    torch.cuda.synchronize()
    eager = (bits(out), bits(dkv), bits(dsc), dape.cpu().numpy().copy())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()
    for fill in (-1, 0):
        out.fill_(fill)
        dkv.fill_(fill)
        dsc.fill_(fill)
        dape.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), eager[0])
        assert np.array_equal(bits(dkv), eager[1]) and np.array_equal(bits(dsc), eager[2])
        assert np.array_equal(dape.cpu().numpy().view(np.uint32), eager[3].view(np.uint32))
    assert csa.csa_device_status() == 0
