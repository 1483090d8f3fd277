"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and lays them out; it computes none of the
update arithmetic.  Both the CUDA path and the fp64 oracle receive the very
same bits from here (the oracle gets exact float64 widenings of them).

Recipes (value distributions follow the workload descriptions: weights
N(0, 0.02), gradients N(0, 1e-3), projector values N(0, 1/sqrt(k)); the
second argument of N is the standard deviation):

* dense tensors: a CPU ``torch.Generator`` seeded per (seed, stream) for
  small cases, or a CUDA generator for full-size layers, drawing fp32
  normals; bf16 tensors are the fp32 draw rounded to nearest-even by
  ``Tensor.to(torch.bfloat16)``.
* projectors: numpy PCG64 seeded per (seed, stream); every row takes k
  distinct column ids uniformly without replacement (a random permutation
  prefix), values N(0, 1/sqrt(k)) in fp32.
"""

import numpy as np
import torch

# --------------------------------------------------------------------------
# seeds
# --------------------------------------------------------------------------


def sub_seed(seed, *stream):
    """Deterministic 63-bit seed for a named sub-stream (layer, tensor, step...)."""
    ss = np.random.SeedSequence([int(seed)] + [int(s) & 0xFFFFFFFF for s in stream])
    return int.from_bytes(ss.generate_state(2, dtype=np.uint32).tobytes(), "little") & ((1 << 63) - 1)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & ((1 << 63) - 1))
    return g


# --------------------------------------------------------------------------
# dense tensors
# --------------------------------------------------------------------------


def normal(shape, std, seed, dtype=torch.float32, device="cpu"):
    """Tensor of N(0, std) draws in ``dtype`` (bf16 = RNE of an fp32 draw)."""
    g = _gen(device, seed)
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(0.0, std, generator=g)
    return x if dtype == torch.float32 else x.to(dtype)


def fill_normal_(t, std, seed, chunk=1 << 28):
    """Fill an existing (possibly huge) tensor with N(0, std) draws, chunk by chunk.

    fp32 draws are rounded to the tensor's dtype.  Chunks use sub-seeds so
    the peak extra memory is one fp32 chunk.
    """
    flat = t.view(-1)
    n = flat.numel()
    for ci, s in enumerate(range(0, n, chunk)):
        e = min(n, s + chunk)
        g = _gen(t.device, sub_seed(seed, ci))
        if t.dtype == torch.float32:
            flat[s:e].normal_(0.0, std, generator=g)
        else:
            tmp = torch.empty(e - s, dtype=torch.float32, device=t.device)
            tmp.normal_(0.0, std, generator=g)
            flat[s:e].copy_(tmp)
            del tmp
    return t


def bf16_bits(t):
    """View a bf16 tensor's storage as uint16 numpy bits (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# projectors
# --------------------------------------------------------------------------


def projector(rows, d, k, seed, replace=False):
    """ELL projector: (idx int32 [rows, k], val float32 [rows, k]).

    Each row draws k column ids from [0, d): without replacement by default
    (a random permutation prefix), with replacement if ``replace``.
    """
    if k > d and not replace:
        raise ValueError("k > d needs replacement")
    rng = np.random.Generator(np.random.PCG64(int(seed) & ((1 << 63) - 1)))
    if replace:
        idx = rng.integers(0, d, size=(rows, k), dtype=np.int64)
    else:
        keys = rng.random((rows, d))
        idx = np.argpartition(keys, k - 1, axis=1)[:, :k] if k < d else np.argsort(keys, axis=1)
        idx = np.take_along_axis(idx, np.argsort(np.take_along_axis(keys, idx, axis=1), axis=1), axis=1)
    val = rng.standard_normal((rows, k)) * (1.0 / np.sqrt(k))
    return idx.astype(np.int32), val.astype(np.float32)


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------

# OPT-1.3B decoder layer: hidden 2048, FFN 8192; QKV fused, out proj, two
# MLP matrices, two LayerNorms (gain, bias).  Biases of the linears are not
# part of the workload description and are left out.
OPT13_LAYER = [
    ("qkv", 3 * 2048 * 2048), ("out", 2048 * 2048),
    ("fc1", 8192 * 2048), ("fc2", 2048 * 8192),
    ("ln1_g", 2048), ("ln1_b", 2048), ("ln2_g", 2048), ("ln2_b", 2048),
]
OPT13_LAYERS = 24

# LLaMA-7B / LLaMA-2-7B decoder layer: hidden 4096, SwiGLU FFN 11008.
LLAMA7_LAYER = [
    ("q", 4096 * 4096), ("k", 4096 * 4096), ("v", 4096 * 4096), ("o", 4096 * 4096),
    ("gate", 11008 * 4096), ("up", 11008 * 4096), ("down", 4096 * 11008),
    ("attn_norm", 4096), ("mlp_norm", 4096),
]
LLAMA7_LAYERS = 32
LLAMA7_VOCAB = 32000

# LLaMA-7B weight-gradient matrices for the projector path: (name, m, n).
LLAMA7_LSP_MATRICES = [
    ("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
    ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008),
]

# Mistral-Large-123B decoder layer: hidden 12288, 96 query heads and 8 KV
# heads of head_dim 128, SwiGLU FFN 28672.
MISTRAL_LAYER = [
    ("q", 12288 * 12288), ("k", 12288 * 1024), ("v", 12288 * 1024), ("o", 12288 * 12288),
    ("gate", 28672 * 12288), ("up", 28672 * 12288), ("down", 12288 * 28672),
    ("attn_norm", 12288), ("mlp_norm", 12288),
]


def llama7_step_order():
    """Tensor groups of the LLaMA-2-7B model in backward (sliding) order.

    LM head, final norm, layers 31..0, embedding: each group is one
    ``[(name, numel), ...]`` list.
    """
    groups = [[("lm_head", LLAMA7_VOCAB * 4096)], [("final_norm", 4096)]]
    for layer in reversed(range(LLAMA7_LAYERS)):
        groups.append([(f"l{layer}.{n}", c) for n, c in LLAMA7_LAYER])
    groups.append([("embed", LLAMA7_VOCAB * 4096)])
    return groups


def layer_numel(layer):
    return sum(c for _, c in layer)
