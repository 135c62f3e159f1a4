"""C-ABI checks that need no GPU: the library loads, exports exactly what
include/csa.h declares, and rejects bad arguments on the host with the
documented status before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_attention_kv_csa_gb300 as csa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"CSA_API\s+[\w\s\*]+?\b(csa_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    decl = declared_symbols()
    assert {"csa_compress_fwd", "csa_compress_bwd", "csa_check_support"} <= decl
    lib = ctypes.CDLL(csa.library_path())
    for name in decl:
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", csa.library_path()], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (csa_\w+)", nm.stdout))
    assert exported == decl


def test_status_strings():
    for code, name in csa.STATUS.items():
        assert csa.csa_status_string(code) == name
    assert csa.csa_status_string(99) == "CSA_ERR_UNKNOWN"


A16 = 1 << 20  # an aligned fake address; validation fails before it is used


@pytest.mark.parametrize("kw,status", [
    (dict(coff=3), 1), (dict(ratio=0), 1), (dict(head_dim=0), 1), (dict(n_seg=-1), 1),
    (dict(capacity=-1), 1), (dict(ratio=129), 2), (dict(head_dim=60), 2), (dict(head_dim=8200), 2),
    (dict(capacity=1 << 30, head_dim=512), 4), (dict(cu=None), 1), (dict(kv=None), 1),
    (dict(out=A16 + 2), 3), (dict(ape=A16 + 4), 3), (dict(cu=A16 + 2), 3),
])
def test_forward_rejects_bad_arguments(kw, status):
    a = dict(kv=A16, score=A16, ape=A16, cu=A16, cc=A16, n_seg=1, ratio=4, coff=2, head_dim=64,
             capacity=8, out=A16)
    a.update(kw)
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_compress_fwd(a["kv"], a["score"], a["ape"], a["cu"], a["cc"], a["n_seg"], a["ratio"],
                             a["coff"], a["head_dim"], a["capacity"], a["out"], stream=0)
    assert ei.value.status == status
    assert csa.csa_last_error_message()


@pytest.mark.parametrize("kw,status", [
    (dict(n_tokens=3), 1), (dict(n_tokens=1 << 22, head_dim=512), 4), (dict(dape=None), 1),
    (dict(dkv=A16 + 8), 3), (dict(grad_out=None), 1), (dict(coff=0), 1),
])
def test_backward_rejects_bad_arguments(kw, status):
    a = dict(kv=A16, score=A16, ape=A16, cu=A16, cc=A16, n_seg=1, ratio=4, coff=2, head_dim=64,
             capacity=8, n_tokens=64, grad_out=A16, dkv=A16, dscore=A16, dape=A16)
    a.update(kw)
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_compress_bwd(a["kv"], a["score"], a["ape"], a["cu"], a["cc"], a["n_seg"], a["ratio"],
                             a["coff"], a["head_dim"], a["capacity"], a["n_tokens"], a["grad_out"], a["dkv"],
                             a["dscore"], a["dape"], stream=0)
    assert ei.value.status == status


def test_forward_capacity_zero_is_a_no_op_without_device():
    # capacity 0 launches nothing, so it succeeds even with no GPU and NULL tensors
    csa.csa_compress_fwd(None, None, None, A16, A16, 1, 4, 2, 64, 0, None, stream=0)


def test_check_support_surface():
    assert csa.csa_check_support(4, 2, 512, 32768, 8256) == 0
    assert csa.csa_check_support(4, 1, 64, 100, 10) == 0
    assert csa.csa_check_support(4, 2, 512, 3, 1) == 1        # fewer tokens than ratio
    assert csa.csa_check_support(4, 2, 512, 3, 0) == 0        # no rows: fine
    assert csa.csa_check_support(4, 2, 512, 1 << 21, 1) == 4  # 2^21 * 1024 >= 2^31
    assert csa.csa_check_support(7, 2, 512, 100, 1) == 0      # generic ratios 1..128
    assert csa.csa_check_support(1, 1, 8, 1, 1) == 0
    assert csa.csa_check_support(129, 1, 512, 1000, 1) == 2   # no kernel beyond 128
    assert csa.csa_check_support(7, 2, 500, 100, 1) == 2      # head_dim % 8
    assert csa.csa_check_support(128, 1, 96, 1000, 1) == 2    # ratio 128: head_dim % 64


@pytest.mark.parametrize("args,status", [
    ((4, 3, 512, 8), 1), ((0, 2, 512, 8), 1), ((4, 2, 0, 8), 1), ((4, 2, 512, -1), 1),
    ((129, 1, 512, 8), 2), ((4, 2, 60, 8), 2), ((128, 1, 96, 8), 2), ((4, 2, 512, 1 << 30), 4),
])
def test_grad_ape_order_rejects_bad_shapes_before_any_device_query(args, status):
    with pytest.raises(csa.CSAError) as ei:
        csa.csa_grad_ape_order(*args)
    assert ei.value.status == status


def test_grad_ape_order_needs_a_device_but_fails_cleanly_without_one():
    import torch
    if torch.cuda.is_available():
        g = csa.csa_grad_ape_order(4, 2, 512, 8256)
        assert g["kind"] == "row_blocks" and g["final_ranges"] == 32
        assert g["partials"] * g["cluster"] == g["blocks"]
    else:
        with pytest.raises(csa.CSAError) as ei:
            csa.csa_grad_ape_order(4, 2, 512, 8256)
        assert ei.value.status == 5  # CSA_ERR_CUDA: no device to query
