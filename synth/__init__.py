"""Seeded synthetic inputs for OUT_PROD and MUL_MAT_ID_BACK.

This module only *makes data*: random numbers, outlier placement, block
quantisation of weights into q8_0 / q4_0 bytes, and expert routing tables.
It holds none of the operations' arithmetic (no dequantisation, no products,
no sums).  Both the CUDA path and the CPU oracle consume the bytes it makes;
neither imports the other.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), state advanced by the golden-ratio
increment 0x9E3779B97F4A7C15.  Uniforms take the top 53 bits; normals use
Box-Muller in float64 (both the cosine and the sine branch, so one pair of
uniforms gives two normals), rounded to float32.

Tensor seeds follow ``seed = 7 * 1000 + tensor_id``.

Outliers (the gradient entries that overflow half precision, seen at up to
1.3e5 in the pages' 0.8B LoRA backward, "metal: OUT_PROD multiplies in float
staging", first comment): exactly ``round(0.002 * numel)`` positions chosen by
a partial Fisher-Yates shuffle, sign by a fair coin, magnitude U(6.6e4, 1.5e5).
"""

from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK = 32                  # elements per q8_0 / q4_0 block
Q8_0_BYTES = 34          # fp16 scale + 32 int8
Q4_0_BYTES = 18          # fp16 scale + 16 bytes of packed nibbles

# ggml's public type ids (the values ggml's enum uses), used on both sides.
TYPE_F32 = 0
TYPE_F16 = 1
TYPE_Q4_0 = 2
TYPE_Q8_0 = 8
TYPE_BF16 = 30

OUTLIER_FRAC = 0.002
OUTLIER_LO = 6.6e4
OUTLIER_HI = 1.5e5

_CHUNK = 1 << 22


def tensor_seed(tensor_id: int, base: int = 7) -> int:
    return base * 1000 + int(tensor_id)


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of the splitmix64 stream for ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform(seed: int, n: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in [0, 1) from the top 53 bits."""
    out = np.empty(n, dtype=np.float64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        z = splitmix64(seed, start + c0, c1 - c0)
        out[c0:c1] = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return out


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float32 normals: Box-Muller in float64, then scaled and rounded once."""
    out = np.empty(n, dtype=np.float32)
    pairs = (n + 1) // 2
    for p0 in range(0, pairs, _CHUNK // 2):
        p1 = min(pairs, p0 + _CHUNK // 2)
        u = uniform(seed, 2 * (p1 - p0), start=2 * p0)
        u1 = 1.0 - u[0::2]                       # (0, 1], so log is finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * np.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = (mean + std * z[: hi - lo]).astype(np.float32)
    return out


def add_outliers(x: np.ndarray, seed: int, frac: float = OUTLIER_FRAC,
                 lo: float = OUTLIER_LO, hi: float = OUTLIER_HI) -> np.ndarray:
    """Replace exactly round(frac*numel) entries of ``x`` (in place, flat order)
    by +-U(lo, hi); positions by partial Fisher-Yates, sign by a fair coin."""
    flat = x.reshape(-1)
    numel = flat.size
    count = int(round(frac * numel))
    if count == 0:
        return x
    u = uniform(seed, 3 * count)
    # partial Fisher-Yates over the index range, kept sparse in a dict
    swapped: dict[int, int] = {}
    picks = np.empty(count, dtype=np.int64)
    for i in range(count):
        j = i + int(u[i] * (numel - i))
        vi = swapped.get(i, i)
        vj = swapped.get(j, j)
        swapped[j] = vi
        picks[i] = vj
    sign = np.where(u[count:2 * count] < 0.5, -1.0, 1.0)
    mag = lo + (hi - lo) * u[2 * count:3 * count]
    flat[picks] = (sign * mag).astype(flat.dtype)
    return x


# ---------------------------------------------------------------------------
# Weight quantisation (producing bytes).  The pages do not say how their test
# weights were quantised; any deterministic quantiser gives valid input bytes.
# Scale per block of 32 consecutive elements along ne0.
# ---------------------------------------------------------------------------

def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """Rows of ``x`` (last dim a multiple of 32) -> uint8 [rows, ne0/32*34].

    Block: little-endian fp16 scale d = fp16(amax/127), then 32 int8
    q = clamp(round-half-away(x/d), -127, 127)."""
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] % QK == 0
    blocks = x.reshape(-1, QK).astype(np.float64)
    amax = np.abs(blocks).max(axis=1)
    d16 = (amax / 127.0).astype(np.float16)
    d = d16.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(d > 0, 1.0 / d, 0.0)
    t = blocks * inv[:, None]
    q = np.clip(np.sign(t) * np.floor(np.abs(t) + 0.5), -127, 127).astype(np.int8)
    out = np.empty((blocks.shape[0], Q8_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)
    out[:, 2:] = q.view(np.uint8)
    return out.reshape(x.shape[:-1] + (x.shape[-1] // QK * Q8_0_BYTES,))


def quantize_q4_0(x: np.ndarray) -> np.ndarray:
    """Rows of ``x`` -> uint8 [rows, ne0/32*18].

    Block: fp16 scale d = fp16(vmax / -8) with vmax the entry of largest
    magnitude (sign kept), then 16 bytes; byte j holds element j in its low
    nibble and element j+16 in its high nibble, each stored as
    clamp(floor(x/d + 8.5), 0, 15)."""
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] % QK == 0
    blocks = x.reshape(-1, QK).astype(np.float64)
    idx = np.abs(blocks).argmax(axis=1)
    vmax = blocks[np.arange(blocks.shape[0]), idx]
    d16 = (vmax / -8.0).astype(np.float16)
    d = d16.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(d != 0, 1.0 / d, 0.0)
    v = np.clip(np.floor(blocks * inv[:, None] + 8.5), 0, 15).astype(np.uint8)
    out = np.empty((blocks.shape[0], Q4_0_BYTES), dtype=np.uint8)
    out[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)
    out[:, 2:] = v[:, :16] | (v[:, 16:] << 4)
    return out.reshape(x.shape[:-1] + (x.shape[-1] // QK * Q4_0_BYTES,))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def row_bytes(type_id: int, ne0: int) -> int:
    if type_id == TYPE_F32:
        return 4 * ne0
    if type_id == TYPE_BF16 or type_id == TYPE_F16:
        return 2 * ne0
    if type_id == TYPE_Q8_0:
        return ne0 // QK * Q8_0_BYTES
    if type_id == TYPE_Q4_0:
        return ne0 // QK * Q4_0_BYTES
    raise ValueError(f"unknown type {type_id}")


def routing_ids(seed: int, n_experts: int, n_used: int, n_tokens: int) -> np.ndarray:
    """int32 [n_tokens, n_used]: per token ``n_used`` distinct experts drawn
    uniformly (partial Fisher-Yates over 0..n_experts-1).  Stored with the
    slot index fastest, i.e. ids[t, i] is slot i of token t."""
    u = uniform(seed, n_tokens * n_used).reshape(n_tokens, n_used)
    out = np.empty((n_tokens, n_used), dtype=np.int32)
    for t in range(n_tokens):
        perm = list(range(n_experts))
        for i in range(n_used):
            j = i + int(u[t, i] * (n_experts - i))
            perm[i], perm[j] = perm[j], perm[i]
            out[t, i] = perm[i]
    return out


# ---------------------------------------------------------------------------
# Workload recipes.  Arrays use C order with ggml's ne0 as the LAST axis, so a
# ggml tensor with ne = {ne0, ne1, ne2, ne3} is a numpy array of shape
# (ne3, ne2, ne1, ne0).
# ---------------------------------------------------------------------------

def make_a(type_id: int, ne: tuple, tensor_id: int, std: float = 1.0,
           base: int = 7) -> np.ndarray:
    """src0 of OUT_PROD: float32 normals, quantised when ``type_id`` asks."""
    ne0, ne1, ne2, ne3 = ne
    x = normal(tensor_seed(tensor_id, base), ne0 * ne1 * ne2 * ne3, std=std)
    x = x.reshape(ne3, ne2, ne1, ne0)
    if type_id == TYPE_F32:
        return x
    if type_id == TYPE_Q8_0:
        return quantize_q8_0(x)
    if type_id == TYPE_Q4_0:
        return quantize_q4_0(x)
    raise ValueError(type_id)


def make_b(ne: tuple, tensor_id: int, std: float = 1.0, outliers: bool = False,
           base: int = 7) -> np.ndarray:
    """src1 of OUT_PROD (the f32 gradient), optionally with outliers."""
    ne0, ne1, ne2, ne3 = ne
    x = normal(tensor_seed(tensor_id, base), ne0 * ne1 * ne2 * ne3, std=std)
    if outliers:
        add_outliers(x, tensor_seed(tensor_id + 500, base))
    return x.reshape(ne3, ne2, ne1, ne0)


# The five workloads, by what they are.
LORA_RANKS = (4, 8, 24)
DENSE_MK = ((1536, 1536), (5120, 5120), (5120, 17408), (17408, 5120))


def single_slice():
    """f32 a [256, 512], b [8, 512], both N(0, 1)."""
    a = make_a(TYPE_F32, (256, 512, 1, 1), 0)
    b = make_b((8, 512, 1, 1), 1)
    return a, b


def lora_rank(r: int):
    """f32 a [2560, 512] ~ N(0,1); b [r, 512] ~ N(0,1)*100 with 0.2% outliers."""
    a = make_a(TYPE_F32, (2560, 512, 1, 1), 10)
    b = make_b((r, 512, 1, 1), 11 + r, std=100.0, outliers=True)
    return a, b


def grouped_heads(n_seq: int):
    """a [128, 512, 4, n_seq], b [128, 512, 16, n_seq], b with outliers."""
    a = make_a(TYPE_F32, (128, 512, 4, n_seq), 20 + n_seq)
    b = make_b((128, 512, 16, n_seq), 22 + n_seq, outliers=True)
    return a, b


def dense_quant(type_id: int, m: int, k: int, n: int = 1024):
    """a = q8_0/q4_0 of N(0, 0.02) [m, k]; b [n, k] ~ N(0,1)*1e3 with outliers."""
    a = make_a(type_id, (m, k, 1, 1), 30, std=0.02)
    b = make_b((n, k, 1, 1), 31, std=1e3, outliers=True)
    return a, b


def moe_back(w_type: int, K: int = 2048, N: int = 768, E: int = 32,
             n_used: int = 8, n_tokens: int = 512):
    """W [K, N, E] ~ N(0, 0.02) (f32, or bf16 bits), ids [n_tokens, n_used],
    g [N, n_used, n_tokens] ~ N(0, 1)."""
    w = normal(tensor_seed(40), K * N * E, std=0.02).reshape(E, N, K)
    if w_type == TYPE_BF16:
        w = to_bf16_bits(w)
    ids = routing_ids(tensor_seed(41), E, n_used, n_tokens)
    g = normal(tensor_seed(42), N * n_used * n_tokens).reshape(n_tokens, n_used, N)
    return w, ids, g
