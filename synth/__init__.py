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
TYPE_Q4_1 = 3
TYPE_Q5_0 = 6
TYPE_Q5_1 = 7
TYPE_Q8_0 = 8
TYPE_Q2_K = 10
TYPE_Q3_K = 11
TYPE_Q4_K = 12
TYPE_Q5_K = 13
TYPE_Q6_K = 14
TYPE_BF16 = 30

QK_K = 256               # elements per K-quant super-block
# (elements, bytes) per block
BLOCK = {TYPE_Q4_0: (32, 18), TYPE_Q4_1: (32, 20), TYPE_Q5_0: (32, 22),
         TYPE_Q5_1: (32, 24), TYPE_Q8_0: (32, 34), TYPE_Q2_K: (256, 84),
         TYPE_Q3_K: (256, 110), TYPE_Q4_K: (256, 144), TYPE_Q5_K: (256, 176),
         TYPE_Q6_K: (256, 210)}
QUANT_TYPES = tuple(BLOCK)

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


def _f16(v):
    """float64 -> (binary16 values as float64, their little-endian bytes)."""
    h = np.asarray(v, dtype=np.float64).astype(np.float16)
    return h.astype(np.float64), h.view(np.uint8).reshape(h.shape + (2,))


def _blocks_of(x, qk):
    x = np.asarray(x, dtype=np.float32)
    assert x.shape[-1] % qk == 0
    return x.reshape(-1, qk).astype(np.float64), x.shape


def _pack_nibbles(v):
    """[blocks, 32] values 0..15 -> [blocks, 16] bytes: byte j holds element j
    (low nibble) and element j + 16 (high nibble)."""
    v = v.astype(np.uint8)
    return v[:, :16] | (v[:, 16:] << 4)


def _safe_div(a, b):
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(b != 0, a / np.where(b != 0, b, 1.0), 0.0)


def quantize_q4_1(x: np.ndarray) -> np.ndarray:
    """Blocks of 32: fp16 d = (max - min)/15, fp16 m = min, then 16 bytes of
    nibbles v = clamp(round((x - m)/d), 0, 15) (q4_0's nibble order)."""
    blocks, shape = _blocks_of(x, 32)
    m, mb = _f16(blocks.min(axis=1))
    d, db = _f16((blocks.max(axis=1) - m) / 15.0)
    v = np.clip(np.rint(_safe_div(blocks - m[:, None], d[:, None])), 0, 15)
    out = np.concatenate([db, mb, _pack_nibbles(v)], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 32 * 20,))


def _q5_pack(v):
    """[blocks, 32] values 0..31 -> (32-bit fifth-bit word as 4 bytes, 16 nibble bytes)."""
    v = v.astype(np.uint32)
    qh = np.zeros(v.shape[0], dtype=np.uint32)
    for j in range(32):
        qh |= ((v[:, j] >> 4) & 1) << j
    return qh.astype("<u4").view(np.uint8).reshape(-1, 4), _pack_nibbles(v & 15)


def quantize_q5_0(x: np.ndarray) -> np.ndarray:
    """Blocks of 32: fp16 d = vmax / -16 (vmax the entry of largest magnitude),
    a 32-bit word of fifth bits, 16 bytes of low nibbles; stored value
    v = clamp(floor(x/d + 16.5), 0, 31), element = d*(v - 16)."""
    blocks, shape = _blocks_of(x, 32)
    vmax = blocks[np.arange(blocks.shape[0]), np.abs(blocks).argmax(axis=1)]
    d, db = _f16(vmax / -16.0)
    v = np.clip(np.floor(_safe_div(blocks, d[:, None]) + 16.5), 0, 31)
    qh, qs = _q5_pack(v)
    out = np.concatenate([db, qh, qs], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 32 * 22,))


def quantize_q5_1(x: np.ndarray) -> np.ndarray:
    """Blocks of 32: fp16 d = (max - min)/31, fp16 m = min, fifth-bit word,
    nibbles; v = clamp(round((x - m)/d), 0, 31), element = d*v + m."""
    blocks, shape = _blocks_of(x, 32)
    m, mb = _f16(blocks.min(axis=1))
    d, db = _f16((blocks.max(axis=1) - m) / 31.0)
    v = np.clip(np.rint(_safe_div(blocks - m[:, None], d[:, None])), 0, 31)
    qh, qs = _q5_pack(v)
    out = np.concatenate([db, mb, qh, qs], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 32 * 24,))


def _pack_scales_k4(sc, mn):
    """[blocks, 8] 6-bit scales and offsets -> [blocks, 12] bytes: sub-blocks
    0..3 in the low six bits of bytes i (scale) and i + 4 (offset); 4..7 as the
    low / high nibble of byte i + 4 with their top two bits in the top bits of
    bytes i - 4 (scale) and i (offset)."""
    sc = sc.astype(np.uint8)
    mn = mn.astype(np.uint8)
    out = np.zeros((sc.shape[0], 12), dtype=np.uint8)
    for i in range(4):
        out[:, i] = (sc[:, i] & 63) | ((sc[:, i + 4] >> 4) << 6)
        out[:, i + 4] = (mn[:, i] & 63) | ((mn[:, i + 4] >> 4) << 6)
        out[:, i + 8] = (sc[:, i + 4] & 15) | ((mn[:, i + 4] & 15) << 4)
    return out


def _quantize_k45(x, levels):
    """Shared part of q4_K (levels 15) and q5_K (levels 31): per 32-element
    sub-block an affine code q in 0..levels with x ~ d*sc*q - dmin*mn, where
    sc and mn are 6-bit and d, dmin the super-block's fp16 scales."""
    blocks, shape = _blocks_of(x, 256)
    sub = blocks.reshape(-1, 8, 32)
    lo = np.minimum(sub.min(axis=2), 0.0)                 # offsets keep 0 reachable
    # offsets and steps rounded up to their 6-bit multiples, so the codes
    # 0..levels always span each sub-block
    dmin, dminb = _f16((-lo).max(axis=1) / 63.0)
    mn = np.clip(np.ceil(_safe_div(-lo, dmin[:, None])), 0, 63)
    off = dmin[:, None] * mn
    scale = (sub.max(axis=2) + off) / levels
    d, db = _f16(scale.max(axis=1) / 63.0)
    sc = np.clip(np.ceil(_safe_div(scale, d[:, None])), 0, 63)
    step = d[:, None] * sc
    q = np.clip(np.rint(_safe_div(sub + off[:, :, None], step[:, :, None])), 0, levels)
    return q.astype(np.uint8), db, dminb, _pack_scales_k4(sc, mn), shape


def _k_nibbles(q):
    """[blocks, 8, 32] codes -> [blocks, 128] bytes: byte 32p + l holds
    sub-block 2p's element l (low nibble) and sub-block 2p+1's (high)."""
    lo = q[:, 0::2, :] & 15
    hi = q[:, 1::2, :] & 15
    return (lo | (hi << 4)).reshape(q.shape[0], 128)


def quantize_q4_k(x: np.ndarray) -> np.ndarray:
    """Super-blocks of 256: fp16 d, fp16 dmin, 12 bytes of 6-bit scales and
    offsets, 128 bytes of 4-bit codes."""
    q, db, dminb, scales, shape = _quantize_k45(x, 15)
    out = np.concatenate([db, dminb, scales, _k_nibbles(q)], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 256 * 144,))


def quantize_q5_k(x: np.ndarray) -> np.ndarray:
    """As q4_K with 5-bit codes: after the scales, 32 bytes whose bit s of
    byte l is the fifth bit of sub-block s's element l, then the nibbles."""
    q, db, dminb, scales, shape = _quantize_k45(x, 31)
    qh = np.zeros((q.shape[0], 32), dtype=np.uint8)
    for sb in range(8):
        qh |= ((q[:, sb, :] >> 4) & 1).astype(np.uint8) << sb
    out = np.concatenate([db, dminb, scales, qh, _k_nibbles(q)], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 256 * 176,))


def quantize_q6_k(x: np.ndarray) -> np.ndarray:
    """Super-blocks of 256 in 16 sub-blocks of 16: int8 scales sc, fp16 d,
    6-bit codes q in 0..63 with x ~ d*sc*(q - 32).  Bytes: 128 of low nibbles,
    64 of 2-bit high parts, 16 scales, d.  Half h, element 32g + l: low nibble
    in byte 64h + l + 32(g%2) (high nibble for g >= 2), high part in bits
    2g..2g+1 of byte 128 + 32h + l, scale 8h + l/16 + 2g."""
    blocks, shape = _blocks_of(x, 256)
    sub = blocks.reshape(-1, 16, 16)
    vmax = np.take_along_axis(sub, np.abs(sub).argmax(axis=2)[:, :, None], 2)[:, :, 0]
    scale = vmax / -32.0
    d, db = _f16(np.abs(scale).max(axis=1) / 127.0)
    # |sc| rounded up, so the codes span the sub-block
    r = _safe_div(scale, d[:, None])
    sc = np.clip(np.sign(r) * np.ceil(np.abs(r)), -128, 127)
    step = d[:, None] * sc
    q = np.clip(np.rint(_safe_div(sub, step[:, :, None])), -32, 31).astype(np.int64) + 32
    q = q.reshape(-1, 256)
    nb = q.shape[0]
    ql = np.zeros((nb, 128), dtype=np.uint8)
    qh = np.zeros((nb, 64), dtype=np.uint8)
    for h in range(2):
        for g in range(4):
            for l in range(32):
                v = q[:, 128 * h + 32 * g + l]
                bi = 64 * h + l + 32 * (g % 2)
                ql[:, bi] |= ((v & 15) << (4 if g >= 2 else 0)).astype(np.uint8)
                qh[:, 32 * h + l] |= (((v >> 4) & 3) << (2 * g)).astype(np.uint8)
    out = np.concatenate([ql, qh, sc.astype(np.int8).view(np.uint8), db], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 256 * 210,))


def quantize_q2_k(x: np.ndarray) -> np.ndarray:
    """Super-blocks of 256 in 16 sub-blocks of 16: scale byte = 4-bit scale
    (low) and 4-bit offset (high), codes 0..3 with x ~ d*sc*q - dmin*mn.
    Bytes: 16 scales, 64 of codes (element 128h + 32g + l in bits 2g..2g+1 of
    byte 32h + l; its scale byte is 8h + 2g + l/16), fp16 d, fp16 dmin."""
    blocks, shape = _blocks_of(x, 256)
    sub = blocks.reshape(-1, 16, 16)
    lo = np.minimum(sub.min(axis=2), 0.0)
    # offsets and steps rounded up (see _quantize_k45)
    dmin, dminb = _f16((-lo).max(axis=1) / 15.0)
    mn = np.clip(np.ceil(_safe_div(-lo, dmin[:, None])), 0, 15)
    off = dmin[:, None] * mn
    scale = (sub.max(axis=2) + off) / 3.0
    d, db = _f16(scale.max(axis=1) / 15.0)
    sc = np.clip(np.ceil(_safe_div(scale, d[:, None])), 0, 15)
    step = d[:, None] * sc
    q = np.clip(np.rint(_safe_div(sub + off[:, :, None], step[:, :, None])), 0, 3)
    q = q.astype(np.uint8).reshape(-1, 256)
    nb = q.shape[0]
    qs = np.zeros((nb, 64), dtype=np.uint8)
    for h in range(2):
        for g in range(4):
            qs[:, 32 * h:32 * h + 32] |= q[:, 128 * h + 32 * g:128 * h + 32 * g + 32] << (2 * g)
    scales = (sc.astype(np.uint8) | (mn.astype(np.uint8) << 4))
    out = np.concatenate([scales, qs, db, dminb], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 256 * 84,))


def quantize_q3_k(x: np.ndarray) -> np.ndarray:
    """Super-blocks of 256 in 16 sub-blocks of 16: signed 6-bit scales (stored
    plus 32), codes q in -4..3 with x ~ d*sc*q.  Bytes: 32 of third bits (bit
    4h + g of byte l, set when q >= 0), 64 of 2-bit parts (q + 4 mod 4, element
    128h + 32g + l in bits 2g..2g+1 of byte 32h + l), 12 of scales (low nibble
    of scale i in byte i for i < 8, high nibble of byte i - 8 for i >= 8; top two
    bits in bits 2*(i/4) of byte 8 + i%4), fp16 d."""
    blocks, shape = _blocks_of(x, 256)
    sub = blocks.reshape(-1, 16, 16)
    vmax = np.take_along_axis(sub, np.abs(sub).argmax(axis=2)[:, :, None], 2)[:, :, 0]
    scale = vmax / -4.0
    d, db = _f16(np.abs(scale).max(axis=1) / 31.0)
    r = _safe_div(scale, d[:, None])
    sc = np.clip(np.sign(r) * np.ceil(np.abs(r)), -32, 31)
    step = d[:, None] * sc
    q = np.clip(np.rint(_safe_div(sub, step[:, :, None])), -4, 3).astype(np.int64) + 4
    q = q.reshape(-1, 256)
    nb = q.shape[0]
    hm = np.zeros((nb, 32), dtype=np.uint8)
    qs = np.zeros((nb, 64), dtype=np.uint8)
    for h in range(2):
        for g in range(4):
            v = q[:, 128 * h + 32 * g:128 * h + 32 * g + 32]
            qs[:, 32 * h:32 * h + 32] |= ((v & 3) << (2 * g)).astype(np.uint8)
            hm |= (((v >> 2) & 1) << (4 * h + g)).astype(np.uint8)
    s6 = (sc.astype(np.int64) + 32).astype(np.uint8)         # 0..63
    scales = np.zeros((nb, 12), dtype=np.uint8)
    for i in range(16):
        low, high = s6[:, i] & 15, s6[:, i] >> 4
        if i < 8:
            scales[:, i] |= low
        else:
            scales[:, i - 8] |= low << 4
        scales[:, 8 + i % 4] |= (high << (2 * (i // 4))).astype(np.uint8)
    out = np.concatenate([hm, qs, scales, db], axis=1)
    return out.reshape(shape[:-1] + (shape[-1] // 256 * 110,))


QUANTIZERS = {}     # filled below, once quantize_q8_0 / quantize_q4_0 exist


def quantize(type_id: int, x: np.ndarray) -> np.ndarray:
    """Rows of x -> the bytes of `type_id` (float16 / bfloat16 bit patterns as
    uint16 for the plain 16-bit types)."""
    if type_id == TYPE_F16:
        return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    if type_id == TYPE_BF16:
        return to_bf16_bits(x)
    return QUANTIZERS[type_id](x)


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
    if type_id in BLOCK:
        qk, nb = BLOCK[type_id]
        return ne0 // qk * nb
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
    return quantize(type_id, x)


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
# (in, out) widths of a 4B layer's seven adapted projections (q, k, v, o,
# gate, up, down): hidden width 2560 as in the rank-r workload, the other
# widths those of a published 4B decoder with 32 query and 8 key-value heads
# of 128 and an MLP of 9728
LAYER_4B_PROJ = ((2560, 4096), (2560, 1024), (2560, 1024), (4096, 2560), (2560, 9728),
                 (2560, 9728), (9728, 2560))
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


QUANTIZERS.update({TYPE_Q4_0: quantize_q4_0, TYPE_Q4_1: quantize_q4_1, TYPE_Q5_0: quantize_q5_0,
                   TYPE_Q5_1: quantize_q5_1, TYPE_Q8_0: quantize_q8_0, TYPE_Q2_K: quantize_q2_k,
                   TYPE_Q3_K: quantize_q3_k, TYPE_Q4_K: quantize_q4_k, TYPE_Q5_K: quantize_q5_k,
                   TYPE_Q6_K: quantize_q6_k})
