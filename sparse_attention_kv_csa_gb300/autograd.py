"""Training-side wrapper: the Compressor as a ``torch.autograd.Function``.

``compress(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, capacity)``
returns ``out`` ([capacity, head_dim] bf16) and, when autograd asks for it,
runs the library's backward, which returns grad_kv, grad_score (bf16, same shape
as kv) and grad_ape (fp32, same shape as ape) ("CSA Fused Compressor", cuDNN
frontend docs, sections Class API and Semantics: the module's forward and its
autograd backward).  The wrapper only checks and marshals arguments: both passes
are the C ABI calls csa_compress_fwd / csa_compress_bwd, on the current stream.

Inputs: kv, score bf16 [n_tokens, coff * head_dim]; ape fp32 [ratio, coff *
head_dim]; cu_seqlens, cu_seqlens_comp int32 [n_seg + 1]; all contiguous on the
same CUDA device.  Gradients flow to kv, score and ape; the offsets and the
static capacity are not differentiable.  The backward rebuilds the softmax from
kv / score / ape (nothing but the inputs is saved), so the saved tensors must not
be modified in place between the two passes (autograd's version counter checks).
"""
import torch

from . import csa_compress_bwd, csa_compress_fwd

__all__ = ["CompressFunction", "compress"]


def _check_inputs(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, require_cuda=True):
    args = (("kv", kv, torch.bfloat16), ("score", score, torch.bfloat16), ("ape", ape, torch.float32),
            ("cu_seqlens", cu_seqlens, torch.int32), ("cu_seqlens_comp", cu_seqlens_comp, torch.int32))
    for name, t, dt in args:
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a tensor" % name)
        if t.dtype != dt:
            raise ValueError("%s must be %s (got %s)" % (name, dt, t.dtype))
    for name, t, _ in args:
        if (require_cuda and not t.is_cuda) or t.device != kv.device:
            raise ValueError("%s must be on kv's CUDA device (got %s)" % (name, t.device))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if kv.dim() != 2 or score.shape != kv.shape:
        raise ValueError("kv and score must be [n_tokens, coff * head_dim] (got %s, %s)"
                         % (tuple(kv.shape), tuple(score.shape)))
    if coff not in (1, 2) or kv.shape[1] % coff:
        raise ValueError("coff must be 1 or 2 and divide kv's width")
    if tuple(ape.shape) != (ratio, kv.shape[1]):
        raise ValueError("ape must be [ratio, coff * head_dim] = [%d, %d] (got %s)"
                         % (ratio, kv.shape[1], tuple(ape.shape)))
    if cu_seqlens.dim() != 1 or cu_seqlens.shape != cu_seqlens_comp.shape or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens and cu_seqlens_comp must both be [n_seg + 1]")


class CompressFunction(torch.autograd.Function):
    """out = Compressor(kv, score, ape); backward through csa_compress_bwd."""

    @staticmethod
    def forward(ctx, kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, capacity):
        _check_inputs(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff)
        head_dim = kv.shape[1] // coff
        n_seg = cu_seqlens.numel() - 1
        out = torch.empty((capacity, head_dim), dtype=torch.bfloat16, device=kv.device)
        csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim, capacity, out)
        ctx.save_for_backward(kv, score, ape, cu_seqlens, cu_seqlens_comp)
        ctx.geometry = (ratio, coff, head_dim, capacity, n_seg)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        kv, score, ape, cu_seqlens, cu_seqlens_comp = ctx.saved_tensors
        ratio, coff, head_dim, capacity, n_seg = ctx.geometry
        if grad_out.dtype != torch.bfloat16:
            raise ValueError("grad_out must be bf16 like out (got %s)" % grad_out.dtype)
        grad_out = grad_out.contiguous()
        dkv = torch.empty_like(kv)
        dscore = torch.empty_like(score)
        dape = torch.empty_like(ape)
        csa_compress_bwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, n_seg, ratio, coff, head_dim, capacity,
                         kv.shape[0], grad_out, dkv, dscore, dape)
        return dkv, dscore, dape, None, None, None, None, None


def compress(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, capacity):
    """The Compressor's forward as a differentiable op (see the module docstring)."""
    return CompressFunction.apply(kv, score, ape, cu_seqlens, cu_seqlens_comp, ratio, coff, capacity)
