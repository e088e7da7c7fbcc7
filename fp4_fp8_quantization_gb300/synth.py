"""Seeded synthetic inputs shaped like mixture-of-experts traffic.

This module only draws random numbers and arranges them: token routing,
ragged row offsets, normal / uniform tensors, random element and scale codes.
It holds none of the quantization or GEMM arithmetic, and both the CUDA path
and the CPU checker consume what it returns.

Recipes (seed 0 unless stated):
* routing: each token picks ``top_k`` distinct experts, uniformly or with
  probabilities p_i proportional to (i + 1)**-s (Zipf); the draw without
  replacement uses the Gumbel-top-k equivalence.  Rows are the (token, slot)
  pairs sorted stably by expert; the groups are the non-empty experts in
  ascending id order.
* bf16 activations: N(0, std) with an optional Bernoulli(p) mask of
  outliers multiplied by a factor.
* FP8 rowwise operands: a bf16 N(0, std) tensor, its per-row (or
  per-channel) amax / 448 as the fp32 scale, and the scaled tensor cast to
  float8_e4m3fn by PyTorch.
* packed FP4 operands: uniformly random nibbles; scale bytes: uniform codes
  in a given range.
"""
import numpy as np
import torch


def topk_ids(num_tokens, top_k, num_experts, seed=0, zipf_s=None):
    """int32 [num_tokens, top_k]: the ``top_k`` distinct experts each token is
    routed to (uniform, or weighted by p_e ~ (e + 1)^-zipf_s)."""
    rng = np.random.default_rng(seed)
    if zipf_s is None:
        logp = np.zeros(num_experts)
    else:
        logp = -zipf_s * np.log(np.arange(1, num_experts + 1, dtype=np.float64))
    keys = logp[None, :] + rng.gumbel(size=(num_tokens, num_experts))
    return np.argpartition(-keys, top_k - 1, axis=1)[:, :top_k].astype(np.int32)


def routing_counts(num_tokens, top_k, num_experts, seed=0, zipf_s=None):
    """Rows per expert when each of ``num_tokens`` tokens is routed to
    ``top_k`` distinct experts (the choices of topk_ids)."""
    chosen = topk_ids(num_tokens, top_k, num_experts, seed, zipf_s)
    return np.bincount(chosen.reshape(-1), minlength=num_experts).astype(np.int64)


def ragged_groups(counts):
    """(a_offsets uint32 [G+1], expert_ids int32 [G]) over the non-empty
    experts, ascending."""
    counts = np.asarray(counts, dtype=np.int64)
    ids = np.nonzero(counts)[0]
    offs = np.concatenate([[0], np.cumsum(counts[ids])])
    return offs.astype(np.uint32), ids.astype(np.int32)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std=1.0, seed=0, device="cpu", outlier_p=0.0,
                outlier_scale=1.0):
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if outlier_p > 0:
        m = torch.rand(shape, generator=g, device=device) < outlier_p
        x = torch.where(m, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def uniform(shape, lo, hi, seed=0, device="cpu"):
    g = _gen(device, seed)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def e4m3_normal(shape, std=1.0, seed=0, device="cpu"):
    """float8_e4m3fn codes of N(0, std) (clamped to the finite range)."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device) * std
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn)


def fp8_rowwise(shape, std=1.0, seed=0, device="cpu"):
    """(codes float8_e4m3fn, scales fp32 [rows]) of an N(0, std) tensor,
    each row divided by its own amax / 448."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device) * std
    x = x.to(torch.bfloat16).float()
    amax = x.abs().amax(dim=-1).clamp_min(1e-30)
    scale = amax / 448.0
    q = (x / scale.unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q, scale


def random_bytes(n, lo=0, hi=255, seed=0, device="cpu"):
    """uint8 [n] uniform on [lo, hi]."""
    g = _gen(device, seed)
    return torch.randint(lo, hi + 1, (n,), generator=g, device=device,
                         dtype=torch.int32).to(torch.uint8)


def random_fp4_packed(shape, seed=0, device="cpu"):
    """Uniformly random packed E2M1 pairs (any byte is two valid codes)."""
    g = _gen(device, seed)
    return torch.randint(0, 256, shape, generator=g, device=device,
                         dtype=torch.int32).to(torch.uint8)
