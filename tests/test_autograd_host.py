"""Argument checks of the autograd wrapper, which raise before any launch (no GPU
needed)."""
import pytest

torch = pytest.importorskip("torch")


def _args(device="cpu", **over):
    a = dict(kv=torch.zeros((16, 8), dtype=torch.bfloat16, device=device),
             score=torch.zeros((16, 8), dtype=torch.bfloat16, device=device),
             ape=torch.zeros((4, 8), dtype=torch.float32, device=device),
             cu=torch.tensor([0, 16], dtype=torch.int32, device=device),
             cc=torch.tensor([0, 4], dtype=torch.int32, device=device))
    a.update(over)
    return a


@pytest.mark.parametrize("over,msg", [
    ({}, "CUDA device"),
    ({"kv": torch.zeros((16, 8), dtype=torch.float16)}, "kv must be torch.bfloat16"),
    ({"ape": torch.zeros((4, 8), dtype=torch.bfloat16)}, "ape must be torch.float32"),
    ({"cu": torch.tensor([0, 16], dtype=torch.int64)}, "cu_seqlens must be torch.int32"),
])
def test_wrapper_rejects_before_launch(over, msg):
    from sparse_attention_kv_csa_gb300.autograd import compress
    a = _args(**over)
    with pytest.raises((ValueError, TypeError), match=msg):
        compress(a["kv"], a["score"], a["ape"], a["cu"], a["cc"], 4, 1, 4)


@pytest.mark.parametrize("over,ratio,coff,msg", [
    ({"score": torch.zeros((16, 4), dtype=torch.bfloat16)}, 4, 1, "kv and score must be"),
    ({}, 4, 3, "coff must be 1 or 2"),
    ({"ape": torch.zeros((2, 8), dtype=torch.float32)}, 4, 1, "ape must be"),
    ({"cc": torch.tensor([0, 4, 4], dtype=torch.int32)}, 4, 1, "cu_seqlens and cu_seqlens_comp"),
])
def test_wrapper_shape_rules(over, ratio, coff, msg):
    from sparse_attention_kv_csa_gb300.autograd import _check_inputs
    a = _args(**over)
    with pytest.raises(ValueError, match=msg):
        _check_inputs(a["kv"], a["score"], a["ape"], a["cu"], a["cc"], ratio, coff, require_cuda=False)


def test_wrapper_accepts_consistent_shapes():
    from sparse_attention_kv_csa_gb300.autograd import _check_inputs
    a = _args()
    _check_inputs(a["kv"], a["score"], a["ape"], a["cu"], a["cc"], 4, 2, require_cuda=False)
