"""Seeded synthetic DiT-MLP workloads (numpy PCG64, BF16 round-to-nearest-even).

The source pages measure Krea 3's MLP on real image edits (a 1 MP reference
latent plus a 4 MP output latent) whose activations and weights are not
available; these generators stand in for them with the shapes and value laws
of the five workloads the library is measured on:

=============  ======================================================================
pr1            x[128][256] ~ N(0,1); W[512][256] ~ N(0,0.02); b[512] ~ N(0,0.01)
dit_up         x[4096][3072] = z*c[k], z ~ N(0,1), c[k] ~ LogNormal(0,0.5) per channel;
               W1[12288][3072] ~ N(0,0.02); b1[12288] ~ N(0,0.01)
dit_down       z[16384][12288] ~ N(0,1) fp32 (the input is MXFP6 of GELU(z));
               W2[3072][12288] ~ N(0,0.01); b2[3072] ~ N(0,0.01)
full_mlp       x[20480][3072] ~ N(0,1); W1[12288][3072], W2[3072][12288] ~ N(0,0.02);
               b1, b2 ~ N(0,0.01)
outlier_mlp    x[20480][4096] ~ Student-t(3); 41 channels (1%, seeded permutation)
               scaled x100; 1% of (row, 32-block) pairs set to +0 (Bernoulli 0.01);
               W1[16384][4096], W2[4096][16384] ~ N(0,0.02); b1, b2 ~ N(0,0.01)
gated_mlp      x[20480][3072] ~ N(0,1); stacked [W_g; W_u][2*8192][3072] ~ N(0,0.02),
               [b_g; b_u][16384] ~ N(0,0.01); W2[3072][8192] ~ N(0,0.02); b2 ~ N(0,0.01)
qkv_proj       x[20480][3072] ~ N(0,1); stacked [W_q; W_k; W_v; W_gate][12288][3072]
               ~ N(0,0.02); b[12288] ~ N(0,0.01)
dit_block      as full_mlp (or gated_mlp's weights), plus the conditioning vectors
               shift, scale, gate [3072] ~ N(0,0.5) and eps = 1e-6
attn_in        x[20480][3072] ~ N(0,1), shift/scale [3072] ~ N(0,0.5), eps = 1e-6,
               stacked [W_q; W_k; W_v; W_gate][12288][3072] ~ N(0,0.02), b ~ N(0,0.01)
attn_out       attention output a[20480][3072] ~ N(0,1), residual x ~ N(0,1) (W2 child),
               W_o[3072][3072] ~ N(0,0.02), b_o ~ N(0,0.01), gate [3072] ~ N(0,0.5)
=============  ======================================================================

Tensors too large to draw on the host (the tests of byte offsets beyond 2^32)
come from a counter-based generator instead, ``hash_bf16_rows`` (numpy, any set of
rows) and ``hash_bf16_fill_`` (torch, a whole tensor on its device). Both compute
the same integer function of (row, column, seed), so a test fills the device
tensor and regenerates only the rows it checks on the host.

Every workload uses seed 0 by default. Each tensor draws from its own child of
SeedSequence(seed), spawned in the fixed order x, W1, b1, W2, b2, channel
scales, masks, shift, scale, gate, so that shrinking one tensor never changes
another (stacked weights draw all their rows from the W1 / b1 child). Values are
drawn in fp32 and rounded to BF16 with round-to-nearest-even; BF16 tensors are
returned as uint16 bit patterns.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_round",
    "bf16_to_f32",
    "hash_bf16_rows",
    "hash_bf16_fill_",
    "workload",
    "pr1",
    "dit_up",
    "dit_down",
    "full_mlp",
    "outlier_mlp",
    "gated_mlp",
    "qkv_proj",
    "dit_block",
    "attn_in",
    "attn_out",
    "WORKLOADS",
]

_ORDER = ("x", "w1", "b1", "w2", "b2", "chan", "mask", "shift", "scale", "gate")


def bf16_round(x) -> np.ndarray:
    """fp32 -> BF16 bit patterns (uint16), round-to-nearest-even. Inputs are finite."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = x.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    """BF16 bit patterns -> fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# Counter-based BF16 values. Element (r, c) takes the key
#   (r * 0x9E3779B1 + c + seed * 0x632BE5AB) mod 2^32
# through Wellons' "lowbias32" integer hash (x ^= x >> 16; x *= 0x7FEB352D;
# x ^= x >> 15; x *= 0x846CA68B; x ^= x >> 16, all mod 2^32); hash bit 31 is the
# sign, bits 24..27 pick the biased exponent 118..133 (magnitudes 2^-9 .. 2^7) and
# bits 0..6 the mantissa, so every value is a finite normal BF16. All arithmetic
# runs on int64 values below 2^63 (the 32-bit products are taken in 16-bit halves),
# so numpy and torch, on any device, compute identical bits. The row multiplier is
# odd, so two rows' keys differ at every column unless the rows are 2^32 apart.
_HASH_ROW = 0x9E3779B1
_HASH_SEED = 0x632BE5AB
_M32 = 0xFFFFFFFF


def _mul32(x, c: int):
    """x * c mod 2^32 for 0 <= x < 2^32, without leaving int64."""
    return (x * (c & 0xFFFF) + (((x * (c >> 16)) & 0xFFFF) << 16)) & _M32


def _hash_bits(r, c, seed: int):
    x = (r * _HASH_ROW + c + seed * _HASH_SEED) & _M32
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return ((x >> 31) << 15) | ((118 + ((x >> 24) & 15)) << 7) | (x & 0x7F)


def hash_bf16_rows(rows, k: int, seed: int = 0) -> np.ndarray:
    """BF16 bit patterns [len(rows)][k] of the counter-based generator, rows by index."""
    r = np.asarray(rows, dtype=np.int64).reshape(-1, 1)
    c = np.arange(k, dtype=np.int64).reshape(1, -1)
    return _hash_bits(r, c, seed).astype(np.uint16)


def hash_bf16_fill_(t, seed: int = 0, row0: int = 0, slab_rows: int = 32768):
    """Fill a contiguous torch.bfloat16 [R][k] tensor in place with the same values
    as hash_bf16_rows(range(row0, row0 + R), k, seed), computed on the tensor's
    device in slabs."""
    import torch

    rows, k = t.shape
    dst = t.view(torch.int16)
    c = torch.arange(k, dtype=torch.int64, device=t.device).reshape(1, -1)
    for lo in range(0, rows, slab_rows):
        hi = min(rows, lo + slab_rows)
        r = torch.arange(row0 + lo, row0 + hi, dtype=torch.int64, device=t.device).reshape(-1, 1)
        bits = _hash_bits(r, c, seed)
        dst[lo:hi].copy_(torch.where(bits >= 32768, bits - 65536, bits).to(torch.int16))
    return t


def _rngs(seed: int) -> dict:
    children = np.random.SeedSequence(seed).spawn(len(_ORDER))
    return {name: np.random.Generator(np.random.PCG64(c)) for name, c in zip(_ORDER, children)}


def _normal_bf16(rng, shape, sigma: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    step = max(1, (1 << 22) // max(1, int(np.prod(shape[1:]))))
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        z = rng.standard_normal((hi - lo,) + tuple(shape[1:]), dtype=np.float32)
        out[lo:hi] = bf16_round(z * np.float32(sigma))
    return out


def pr1(seed: int = 0, M: int = 128, K: int = 256, N: int = 512) -> dict:
    """Single GEMM: activations x[M][K], weight w[N][K], bias b[N] (BF16 bits)."""
    r = _rngs(seed)
    return {
        "x": _normal_bf16(r["x"], (M, K), 1.0),
        "w": _normal_bf16(r["w1"], (N, K), 0.02),
        "b": _normal_bf16(r["b1"], (N,), 0.01),
    }


def dit_up(seed: int = 0, M: int = 4096, d: int = 3072, ff: int = 12288) -> dict:
    """Up-projection: x = z * c[channel] with log-normal channel scales."""
    r = _rngs(seed)
    chan = r["chan"].lognormal(0.0, 0.5, size=d).astype(np.float32)
    x = np.empty((M, d), dtype=np.uint16)
    step = max(1, (1 << 22) // d)
    for lo in range(0, M, step):
        hi = min(M, lo + step)
        z = r["x"].standard_normal((hi - lo, d), dtype=np.float32)
        x[lo:hi] = bf16_round(z * chan[None, :])
    return {
        "x": x,
        "w": _normal_bf16(r["w1"], (ff, d), 0.02),
        "b": _normal_bf16(r["b1"], (ff,), 0.01),
        "chan": chan,
    }


def dit_down(seed: int = 0, M: int = 16384, ff: int = 12288, d: int = 3072) -> dict:
    """Down-projection: z[M][ff] ~ N(0,1) fp32 (input is MXFP6 of GELU(z)), W2, b2."""
    r = _rngs(seed)
    z = np.empty((M, ff), dtype=np.float32)
    step = max(1, (1 << 22) // ff)
    for lo in range(0, M, step):
        hi = min(M, lo + step)
        z[lo:hi] = r["x"].standard_normal((hi - lo, ff), dtype=np.float32)
    return {
        "z": z,
        "w": _normal_bf16(r["w2"], (d, ff), 0.01),
        "b": _normal_bf16(r["b2"], (d,), 0.01),
    }


def full_mlp(seed: int = 0, M: int = 20480, d: int = 3072, ff: int = 12288) -> dict:
    """Full DiT MLP block: x, W1, b1, W2, b2 (BF16 bits)."""
    r = _rngs(seed)
    return {
        "x": _normal_bf16(r["x"], (M, d), 1.0),
        "w1": _normal_bf16(r["w1"], (ff, d), 0.02),
        "b1": _normal_bf16(r["b1"], (ff,), 0.01),
        "w2": _normal_bf16(r["w2"], (d, ff), 0.02),
        "b2": _normal_bf16(r["b2"], (d,), 0.01),
    }


def outlier_mlp(seed: int = 0, M: int = 20480, d: int = 4096, ff: int = 16384) -> dict:
    """Outlier-heavy wide MLP: heavy-tailed activations, hot channels, zero blocks."""
    r = _rngs(seed)
    n_hot = int(round(0.01 * d))
    hot = np.sort(r["chan"].permutation(d)[:n_hot])
    gain = np.ones(d, dtype=np.float32)
    gain[hot] = 100.0
    x = np.empty((M, d), dtype=np.uint16)
    step = max(1, (1 << 21) // d)
    for lo in range(0, M, step):
        hi = min(M, lo + step)
        t = r["x"].standard_t(3.0, size=(hi - lo, d)).astype(np.float32)
        t *= gain[None, :]
        zero = r["mask"].random((hi - lo, d // 32)) < 0.01
        t.reshape(hi - lo, d // 32, 32)[zero] = 0.0
        x[lo:hi] = bf16_round(t)
    return {
        "x": x,
        "w1": _normal_bf16(r["w1"], (ff, d), 0.02),
        "b1": _normal_bf16(r["b1"], (ff,), 0.01),
        "w2": _normal_bf16(r["w2"], (d, ff), 0.02),
        "b2": _normal_bf16(r["b2"], (d,), 0.01),
        "hot_channels": hot,
    }


def gated_mlp(seed: int = 0, M: int = 20480, d: int = 3072, ff: int = 8192) -> dict:
    """SwiGLU MLP: x, stacked gate/up weight wgu [2 ff][d] (gate rows first) and
    bias bgu [2 ff], W2 [d][ff], b2 (BF16 bits). ff = 8192 is 2/3 of 4d, so the
    three GEMMs do the same work as the GELU MLP's two at ff = 4d."""
    r = _rngs(seed)
    return {
        "x": _normal_bf16(r["x"], (M, d), 1.0),
        "wgu": _normal_bf16(r["w1"], (2 * ff, d), 0.02),
        "bgu": _normal_bf16(r["b1"], (2 * ff,), 0.01),
        "w2": _normal_bf16(r["w2"], (d, ff), 0.02),
        "b2": _normal_bf16(r["b2"], (d,), 0.01),
    }


def qkv_proj(seed: int = 0, M: int = 20480, d: int = 3072, stack: int = 4) -> dict:
    """Stacked query/key/value/attention-gate projection: x [M][d], w [4d][d], b [4d]."""
    r = _rngs(seed)
    return {
        "x": _normal_bf16(r["x"], (M, d), 1.0),
        "w": _normal_bf16(r["w1"], (stack * d, d), 0.02),
        "b": _normal_bf16(r["b1"], (stack * d,), 0.01),
    }


def dit_block(seed: int = 0, M: int = 20480, d: int = 3072, ff: int | None = None,
              activation: str = "gelu") -> dict:
    """MLP half of a DiT block: x, conditioning shift/scale/gate [d], eps, the up
    weight w_up (W1 [ff][d] for "gelu", stacked [W_g; W_u] [2 ff][d] for "swiglu"),
    b_up, W2 [d][ff], b2. ff defaults to 4d (gelu) or 8d/3 (swiglu)."""
    if ff is None:
        ff = 4 * d if activation == "gelu" else (8 * d) // 3
    r = _rngs(seed)
    rows_up = ff if activation == "gelu" else 2 * ff
    return {
        "x": _normal_bf16(r["x"], (M, d), 1.0),
        "w_up": _normal_bf16(r["w1"], (rows_up, d), 0.02),
        "b_up": _normal_bf16(r["b1"], (rows_up,), 0.01),
        "w2": _normal_bf16(r["w2"], (d, ff), 0.02),
        "b2": _normal_bf16(r["b2"], (d,), 0.01),
        "shift": _normal_bf16(r["shift"], (d,), 0.5),
        "scale": _normal_bf16(r["scale"], (d,), 0.5),
        "gate": _normal_bf16(r["gate"], (d,), 0.5),
        "eps": 1e-6,
        "activation": activation,
    }


def attn_in(seed: int = 0, M: int = 20480, d: int = 3072) -> dict:
    """Attention input of a DiT block: x, shift, scale, eps (RMSNorm + modulation),
    then the stacked query/key/value/attention-gate weight w [4d][d] and bias b."""
    r = _rngs(seed)
    return {
        "x": _normal_bf16(r["x"], (M, d), 1.0),
        "shift": _normal_bf16(r["shift"], (d,), 0.5),
        "scale": _normal_bf16(r["scale"], (d,), 0.5),
        "eps": 1e-6,
        "w": _normal_bf16(r["w1"], (4 * d, d), 0.02),
        "b": _normal_bf16(r["b1"], (4 * d,), 0.01),
    }


def attn_out(seed: int = 0, M: int = 20480, d: int = 3072) -> dict:
    """Attention output projection with gate and residual: the attention output a,
    the block input x (the residual), W_o [d][d], b_o, gate [d]."""
    r = _rngs(seed)
    return {
        "a": _normal_bf16(r["x"], (M, d), 1.0),
        "x": _normal_bf16(r["w2"], (M, d), 1.0),
        "w": _normal_bf16(r["w1"], (d, d), 0.02),
        "b": _normal_bf16(r["b1"], (d,), 0.01),
        "gate": _normal_bf16(r["gate"], (d,), 0.5),
    }


WORKLOADS = {
    "pr1": pr1,
    "dit_up": dit_up,
    "dit_down": dit_down,
    "full_mlp": full_mlp,
    "outlier_mlp": outlier_mlp,
    "gated_mlp": gated_mlp,
    "qkv_proj": qkv_proj,
    "dit_block": dit_block,
    "attn_in": attn_in,
    "attn_out": attn_out,
}


def workload(name: str, **kw) -> dict:
    """Generate a named workload (see the table in this module's docstring)."""
    return WORKLOADS[name](**kw)
