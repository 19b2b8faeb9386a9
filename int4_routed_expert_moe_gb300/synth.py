"""Seeded synthetic inputs for the routed INT4-expert MoE FFN.

This module only draws random numbers and lays them out in arrays. It holds
none of the method's arithmetic (no dequantisation, routing, activation or
combine): both the CPU oracle and the CUDA library consume what it returns.

Storage convention of one expert (the canonical form, consumed unchanged by the
library's expert block):

* ``qp_gate`` uint8 [I][H/2], ``qp_up`` uint8 [I][H/2], ``qp_down`` uint8 [H][I/2]
  -- packed 4-bit codes of the weight matrices W_g [I][H], W_u [I][H],
  W_d [H][I]; byte c of a row holds element 2c in its low nibble and element
  2c+1 in its high nibble. Uniform random bytes give uniform codes 0..15.
* ``s_*`` / ``z_*`` float16 [rows][cols/g] -- one scale and one zero point for
  each run of g consecutive elements along a row (the reduction axis).

Distributions follow the workloads the pages measure (OLMoE-like 64-expert
top-8 layers, a 512-expert top-10 stack): activations N(0,1) in FP16, router
logits FP32 (N(0,1), U(0,1), or Zipf-popular via the Gumbel-top-k trick),
scales U(1e-3, 1e-2) in FP16, zero point 8.
"""
from __future__ import annotations

import numpy as np

# Workloads. Names say what they are; sizes are the ones each case runs at.
WORKLOADS = {
    "tiny_layer": dict(L=1, H=256, I=128, E=8, k=2, g=64, renorm=True, T=4,
                       logits="normal"),
    "olmoe_decode": dict(L=16, H=2048, I=1024, E=64, k=8, g=128, renorm=False,
                         T=1, steps=128, logits="normal"),
    "olmoe_partial": dict(L=16, H=2048, I=1024, E=64, k=8, g=128, renorm=False,
                          T=1, steps=128, seqs=12, warm_seqs=1, C=30,
                          decay=0.9, logits="zipf", alpha=1.0),
    "olmoe_prefill": dict(L=16, H=2048, I=1024, E=64, k=8, g=128, renorm=False,
                          T=512, logits="uniform", Ts=2048, Is=4096),
    "large_fanout": dict(L=48, H=2048, I=512, E=512, k=10, g=128, renorm=True,
                         T=(1, 16, 256), logits="zipf", alpha=1.1),
    # Qwen-like routed stack: 60 experts, top-4 without renormalisation,
    # expert intermediate 1408, 24 layers.
    "qwen_decode": dict(L=24, H=2048, I=1408, E=60, k=4, g=128, renorm=False,
                        T=1, steps=128, logits="normal"),
}

BASE_SEED = 20261202


def rng_for(*key: int) -> np.random.Generator:
    """Independent PCG64 stream for a tuple of integer keys."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [int(v) & 0xFFFFFFFF for v in key])))


def expert_arrays(seed: int, layer: int, expert: int, H: int, I: int, g: int,
                  zero: str = "eight", codes: str = "uniform") -> dict:
    """Canonical arrays of one expert, seeded by (seed, layer, expert).

    ``zero``: "eight" (z = 8.0), "int" (random integer 0..15) or "frac"
    (random FP16 in [0, 15]). ``codes``: "uniform" random bytes.
    """
    r = rng_for(seed, layer, expert)

    def packed(rows, cols):
        return r.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)

    def scales(rows, cols):
        return r.uniform(1e-3, 1e-2, size=(rows, cols // g)).astype(np.float16)

    def zeros(rows, cols):
        shape = (rows, cols // g)
        if zero == "eight":
            return np.full(shape, 8.0, dtype=np.float16)
        if zero == "int":
            return r.integers(0, 16, size=shape).astype(np.float16)
        if zero == "frac":
            return r.uniform(0.0, 15.0, size=shape).astype(np.float16)
        raise ValueError(zero)

    out = {}
    out["qp_gate"] = packed(I, H)
    out["qp_up"] = packed(I, H)
    out["qp_down"] = packed(H, I)
    out["s_gate"], out["z_gate"] = scales(I, H), zeros(I, H)
    out["s_up"], out["z_up"] = scales(I, H), zeros(I, H)
    out["s_down"], out["z_down"] = scales(H, I), zeros(H, I)
    return out


def activations(seed: int, tag: int, T: int, H: int) -> np.ndarray:
    """x ~ N(0,1) rounded to FP16, shape [T][H]."""
    return rng_for(seed, 0x7A, tag).standard_normal((T, H)).astype(np.float16)


def logits_normal(seed: int, tag: int, T: int, E: int) -> np.ndarray:
    return rng_for(seed, 0x10, tag).standard_normal((T, E)).astype(np.float32)


def logits_uniform(seed: int, tag: int, T: int, E: int) -> np.ndarray:
    return rng_for(seed, 0x11, tag).uniform(0.0, 1.0, (T, E)).astype(np.float32)


def zipf_ranks(seed: int, layer: int, E: int) -> np.ndarray:
    """Popularity rank (1 = most popular) of every expert of a layer."""
    perm = rng_for(seed, 0x20, layer).permutation(E)
    ranks = np.empty(E, dtype=np.int64)
    ranks[perm] = np.arange(1, E + 1)
    return ranks


def logits_zipf(seed: int, layer: int, tag: int, T: int, E: int,
                alpha: float) -> np.ndarray:
    """Logits whose top-k is a draw without replacement with P(e) ~ rank^-alpha.

    l_e = -alpha * ln(rank_e) + G_e with G_e ~ Gumbel(0, 1) (Gumbel-top-k).
    """
    ranks = zipf_ranks(seed, layer, E)
    gum = rng_for(seed, 0x21, layer, tag).gumbel(0.0, 1.0, (T, E))
    return (-alpha * np.log(ranks)[None, :] + gum).astype(np.float32)


def logits_for(wl: dict, seed: int, layer: int, tag: int, T: int) -> np.ndarray:
    kind = wl["logits"]
    E = wl["E"]
    if kind == "normal":
        return logits_normal(seed, layer * 1_000_003 + tag, T, E)
    if kind == "uniform":
        return logits_uniform(seed, layer * 1_000_003 + tag, T, E)
    if kind == "zipf":
        return logits_zipf(seed, layer, tag, T, E, wl["alpha"])
    raise ValueError(kind)


def shared_weights(seed: int, H: int, Is: int) -> dict:
    """FP16 weights of the dense non-routed SwiGLU FFN, scaled to keep O(1) outputs."""
    r = rng_for(seed, 0x30)
    wg = (r.standard_normal((Is, H)) / np.sqrt(H)).astype(np.float16)
    wu = (r.standard_normal((Is, H)) / np.sqrt(H)).astype(np.float16)
    wd = (r.standard_normal((H, Is)) / np.sqrt(Is)).astype(np.float16)
    return {"wg": wg, "wu": wu, "wd": wd}


def pack_codes(q: np.ndarray) -> np.ndarray:
    """Pack an explicit code matrix [rows][cols] (values 0..15) into bytes.

    Test helper for hand-made cases: byte c = q[2c] | q[2c+1] << 4. This is the
    storage convention, not the method.
    """
    q = np.asarray(q, dtype=np.uint8)
    assert q.ndim == 2 and q.shape[1] % 2 == 0 and int(q.max(initial=0)) < 16
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def block_layout(H: int, I: int, g: int) -> dict:
    """Byte geometry of one expert block as the library's header documents it:
    gate/up rows [q_gate | q_up | per-group quads (s_gate, z_gate, s_up, z_up)]
    and down rows [q_down | per-group pairs (s_down, z_down)], each row padded
    to 16 bytes. Sizes only."""
    ggu, gd = H // g, I // g
    gu_row = (H + 8 * ggu + 15) // 16 * 16
    d_row = (I // 2 + 4 * gd + 15) // 16 * 16
    return {"gu_codes": {"qp_gate": (0, H // 2), "qp_up": (H // 2, H)},
            "gu_sz": (H, ggu, ("s_gate", "z_gate", "s_up", "z_up")),
            "d_codes": {"qp_down": (0, I // 2)},
            "d_sz": (I // 2, gd, ("s_down", "z_down")),
            "gu_row": gu_row, "d_row": d_row, "d_offset": I * gu_row,
            "total": I * gu_row + H * d_row}


def device_pool(n_blocks: int, H: int, I: int, g: int, seed: int, device="cuda",
                chunk: int = 64):
    """A pool of n_blocks expert blocks generated on the device with torch's
    CUDA generator (seeded): uniform code bytes, scales U(1e-3, 1e-2) in FP16,
    zero points 8, padding 0. Same distributions as expert_arrays; used where
    host generation of many gigabytes would be too slow."""
    import torch
    lay = block_layout(H, I, g)
    bb = lay["total"]
    pool = torch.zeros((n_blocks, bb), dtype=torch.uint8, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    for b0 in range(0, n_blocks, chunk):
        b1 = min(n_blocks, b0 + chunk)
        n = b1 - b0
        blk = pool[b0:b1]
        sections = ((blk[:, :lay["d_offset"]].view(n, I, lay["gu_row"]), lay["gu_codes"], lay["gu_sz"]),
                    (blk[:, lay["d_offset"]:].view(n, H, lay["d_row"]), lay["d_codes"], lay["d_sz"]))
        for view, codes, (start, groups, names) in sections:
            rows = view.shape[1]
            for lo, hi in codes.values():
                view[:, :, lo:hi] = torch.randint(0, 256, (n, rows, hi - lo), dtype=torch.uint8,
                                                  device=device, generator=gen)
            vals = torch.empty((n, rows, groups, len(names)), dtype=torch.float16, device=device)
            for i, name in enumerate(names):
                if name.startswith("s"):
                    v = torch.empty((n, rows, groups), dtype=torch.float32, device=device)
                    v.uniform_(1e-3, 1e-2, generator=gen)
                    vals[:, :, :, i] = v.to(torch.float16)
                else:
                    vals[:, :, :, i] = 8.0
            view[:, :, start:start + groups * len(names) * 2] = vals.view(torch.uint8).view(n, rows, -1)
    return pool


def arrays_from_block(block, H: int, I: int, g: int) -> dict:
    """Canonical arrays of one expert read out of a block's bytes (host numpy)."""
    lay = block_layout(H, I, g)
    b = np.asarray(block, dtype=np.uint8)
    gu = b[:lay["d_offset"]].reshape(I, lay["gu_row"])
    d = b[lay["d_offset"]:lay["total"]].reshape(H, lay["d_row"])
    out = {}
    for view, codes, (start, groups, names) in ((gu, lay["gu_codes"], lay["gu_sz"]),
                                                (d, lay["d_codes"], lay["d_sz"])):
        for name, (lo, hi) in codes.items():
            out[name] = np.ascontiguousarray(view[:, lo:hi])
        sz = np.ascontiguousarray(view[:, start:start + groups * len(names) * 2]).view(np.float16)
        sz = sz.reshape(view.shape[0], groups, len(names))
        for i, name in enumerate(names):
            out[name] = np.ascontiguousarray(sz[:, :, i])
    return out
