"""The autograd wrapper (sparse_attention_kv_csa_gb300.autograd) against the C ABI
calls it wraps and against the fp32 oracle: the forward value, and the gradients
autograd delivers to kv, score and ape for a loss built on the output."""
import numpy as np
import pytest

import csa_workloads as w
import oracle
from gpu_util import Dev, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import sparse_attention_kv_csa_gb300 as m
    return m


def _leaf(t, dtype):
    return t.view(dtype).clone().requires_grad_(True)


@pytest.mark.parametrize("name,ratio,coff,head_dim,lens", [
    ("ag_tiny", 4, 2, 64, [37, 64]),
    ("ag_stream", 4, 2, 512, [1000, 4, 333]),
    ("ag_r128", 128, 1, 128, [700, 129]),
])
def test_autograd_matches_the_abi(csa, name, ratio, coff, head_dim, lens):
    import torch
    from sparse_attention_kv_csa_gb300.autograd import compress
    c = w.make_case(name, ratio, coff, head_dim, lens, extra_rows=3, seed=21)
    d = Dev(c)
    kv = _leaf(d.kv, torch.bfloat16)
    sc = _leaf(d.score, torch.bfloat16)
    ape = d.ape.clone().requires_grad_(True)
    out = compress(kv, sc, ape, d.cu, d.cc, ratio, coff, c.capacity)
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (c.capacity, head_dim)
    out.backward(d.g.view(torch.bfloat16))
    torch.cuda.synchronize()
    want_out = run_fwd(d, csa)
    want_dkv, want_dsc, want_dape = run_bwd(d, csa)
    assert np.array_equal(out.detach().cpu().view(torch.int16).numpy().view(np.uint16), want_out)
    assert np.array_equal(kv.grad.cpu().view(torch.int16).numpy().view(np.uint16), want_dkv)
    assert np.array_equal(sc.grad.cpu().view(torch.int16).numpy().view(np.uint16), want_dsc)
    assert np.array_equal(ape.grad.cpu().numpy().view(np.uint32), want_dape.view(np.uint32))
    if ratio == 4:  # the ratio-4 kernels are bitwise equal to the fp32 oracle
        assert np.array_equal(want_out, oracle.case_fwd_f32(c))


def test_autograd_loss_on_the_output(csa):
    """loss = sum(out * W): autograd hands the backward grad_out = bf16(W)."""
    import torch
    from sparse_attention_kv_csa_gb300.autograd import compress
    c = w.make_case("ag_loss", 4, 2, 128, [96, 41], seed=5)
    d = Dev(c)
    kv = _leaf(d.kv, torch.bfloat16)
    sc = _leaf(d.score, torch.bfloat16)
    ape = d.ape.clone().requires_grad_(True)
    W = torch.from_numpy(np.random.default_rng(1).standard_normal((c.capacity, c.head_dim)).astype(np.float32))
    W = W.cuda().to(torch.bfloat16)
    out = compress(kv, sc, ape, d.cu, d.cc, 4, 2, c.capacity)
    (out * W).sum().backward()
    d.g = W.view(torch.int16).contiguous()
    want_dkv, want_dsc, want_dape = run_bwd(d, csa)
    assert np.array_equal(kv.grad.cpu().view(torch.int16).numpy().view(np.uint16), want_dkv)
    assert np.array_equal(sc.grad.cpu().view(torch.int16).numpy().view(np.uint16), want_dsc)
    assert np.array_equal(ape.grad.cpu().numpy().view(np.uint32), want_dape.view(np.uint32))
    assert csa.csa_device_status() == 0
