"""Counter-based random streams and the five benchmark workloads.

Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: draw i of stream (seed, tag) is mix64(base + (i + 1) * GOLDEN),
base = mix64(seed << 32 | tag).  Uniforms take the top 53 bits; normals use
the Box-Muller transform (both outputs of each pair).  Everything is drawn in
fp64 and rounded to fp32 / fp16 at the end.

Workloads (the task's five configurations; the log pages measured them on a
"7B" q4_K_m model prefill, which these synthetic tensors stand in for):
  0 q6_K tiny          od=256   id=512    nt=16
  1 q4_K q-proj        od=3584  id=3584   nt=512
  2 q6_K q-proj        od=3584  id=3584   nt=512
  3 q4_K FFN up/gate   od=18944 id=3584   nt=2630  X ~ N(0, 1.5)
  4 q6_K FFN down      od=3584  id=18944  nt=2630  X ~ N(0,1), 1% outliers x20
q6_K blocks: ql/qh bytes uniform, int8 sub-block scales uniform in [-32, 31]
(the workloads' recipe), fp16 d = fp16_rn(U[1e-4, 1e-3]).  scales="int8"
spreads the scales the way the format is usually encoded instead, the
sub-block of largest magnitude at -128 and the rest in proportion: per
super-block 16 magnitudes U[0.3, 1] with random signs s_i, sc_i =
clip(rint(-128 s_i / s_k), -128, 127), k the largest |s_i| (most |sc| then
exceed 64, which the GEMM handles with a two-plane operand).  q4_K blocks: qs bytes uniform, the 12
packed scale/min bytes uniform (every 6-bit field is then uniform in [0, 63]),
fp16 d and dmin = fp16_rn(U[1e-4, 1e-3]).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream tags (one independent stream per field)
TAG_X = 1
TAG_X_OUTLIER = 2
TAG_W_BYTES = 3
TAG_W_SCALE = 4
TAG_W_D = 5
TAG_W_DMIN = 6
TAG_W_SCALE_SIGN = 7


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """n draws (uint64) of stream (seed, tag), starting at draw `offset`."""
    with np.errstate(over="ignore"):
        base = _mix(np.array([((seed & 0xFFFFFFFF) << 32) | (tag & 0xFFFFFFFF)],
                             dtype=np.uint64))[0]
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(base + ctr * GOLDEN)


def uniform01(seed: int, tag: int, n: int) -> np.ndarray:
    """U[0, 1) in fp64 (53-bit)."""
    return (splitmix64(seed, tag, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_bytes(seed: int, tag: int, n: int) -> np.ndarray:
    """n uniform bytes: the little-endian bytes of ceil(n/8) draws."""
    w = splitmix64(seed, tag, (n + 7) // 8)
    return w.astype("<u8").view(np.uint8)[:n].copy()


def normal(seed: int, tag: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma^2) in fp64 by Box-Muller; 2 normals per pair of uniforms."""
    m = (n + 1) // 2
    u = uniform01(seed, tag, 2 * m)
    u1 = 1.0 - u[0::2]                  # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n] * sigma


def f16_uniform(seed: int, tag: int, n: int, lo: float, hi: float) -> np.ndarray:
    """fp16 bit patterns of fp16_rn(U[lo, hi])."""
    u = lo + (hi - lo) * uniform01(seed, tag, n)
    return u.astype(np.float16).view(np.uint16)


def q6k_blocks(seed: int, nblk: int, scales: str = "small") -> np.ndarray:
    """nblk packed 210-byte q6_K blocks: ql[128] qh[64] sc[16] d(fp16)."""
    out = np.empty((nblk, 210), dtype=np.uint8)
    out[:, 0:192] = uniform_bytes(seed, TAG_W_BYTES, nblk * 192).reshape(nblk, 192)
    if scales == "small":
        sc = (uniform_bytes(seed, TAG_W_SCALE, nblk * 16).astype(np.int16) & 63) - 32
    elif scales == "int8":
        mag = 0.3 + 0.7 * uniform01(seed, TAG_W_SCALE, nblk * 16).reshape(nblk, 16)
        sign = np.where(uniform_bytes(seed, TAG_W_SCALE_SIGN, nblk * 16).reshape(nblk, 16) & 1, -1.0, 1.0)
        s = mag * sign
        sk = s[np.arange(nblk), np.argmax(mag, axis=1)][:, None]
        sc = np.clip(np.rint(-128.0 * s / sk), -128, 127).astype(np.int16)
    else:
        raise ValueError(f"q6_K scales: {scales!r}")
    out[:, 192:208] = sc.astype(np.int8).view(np.uint8).reshape(nblk, 16)
    d = f16_uniform(seed, TAG_W_D, nblk, 1e-4, 1e-3)
    out[:, 208:210] = d.astype("<u2").view(np.uint8).reshape(nblk, 2)
    return out


def q4k_blocks(seed: int, nblk: int) -> np.ndarray:
    """nblk packed 144-byte q4_K blocks: d dmin (fp16) scales[12] qs[128]."""
    out = np.empty((nblk, 144), dtype=np.uint8)
    out[:, 0:2] = f16_uniform(seed, TAG_W_D, nblk, 1e-4, 1e-3).astype("<u2").view(
        np.uint8).reshape(nblk, 2)
    out[:, 2:4] = f16_uniform(seed, TAG_W_DMIN, nblk, 1e-4, 1e-3).astype("<u2").view(
        np.uint8).reshape(nblk, 2)
    out[:, 4:16] = uniform_bytes(seed, TAG_W_SCALE, nblk * 12).reshape(nblk, 12)
    out[:, 16:144] = uniform_bytes(seed, TAG_W_BYTES, nblk * 128).reshape(nblk, 128)
    return out


@dataclass(frozen=True)
class Config:
    index: int
    name: str
    qtype: str          # "q4_K" | "q6_K"
    od: int
    id: int
    nt: int
    seed: int
    sigma: float = 1.0
    outlier_p: float = 0.0
    outlier_scale: float = 1.0

    @property
    def ops(self) -> int:
        return 2 * self.nt * self.od * self.id


CONFIGS = [
    Config(0, "q6_K_tiny_256x512_nt16", "q6_K", 256, 512, 16, 0),
    Config(1, "q4_K_qproj_3584x3584_nt512", "q4_K", 3584, 3584, 512, 1),
    Config(2, "q6_K_qproj_3584x3584_nt512", "q6_K", 3584, 3584, 512, 2),
    Config(3, "q4_K_ffn_up_18944x3584_nt2630", "q4_K", 18944, 3584, 2630, 3, sigma=1.5),
    Config(4, "q6_K_ffn_down_3584x18944_nt2630", "q6_K", 3584, 18944, 2630, 4,
           outlier_p=0.01, outlier_scale=20.0),
]


def config_by_name(name: str) -> Config:
    for c in CONFIGS:
        if c.name == name or str(c.index) == str(name):
            return c
    raise KeyError(name)


def weights(qtype: str, od: int, id_: int, seed: int, q6_scales: str = "small") -> np.ndarray:
    """Packed weight rows: od x (id/256) blocks, row-major, as a flat uint8 array."""
    nblk = od * (id_ // 256)
    blk = q6k_blocks(seed, nblk, q6_scales) if qtype == "q6_K" else q4k_blocks(seed, nblk)
    return blk.reshape(-1)


def activations(nt: int, id_: int, seed: int, sigma: float = 1.0,
                outlier_p: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    """fp32 activations (nt, id): N(0, sigma^2); each entry independently
    multiplied by outlier_scale with probability outlier_p."""
    x = normal(seed, TAG_X, nt * id_, sigma)
    if outlier_p > 0.0:
        u = uniform01(seed, TAG_X_OUTLIER, nt * id_)
        x = np.where(u < outlier_p, x * outlier_scale, x)
    return x.astype(np.float32).reshape(nt, id_)


def config_inputs(cfg: Config):
    """(W flat uint8, X fp32 (nt, id)) for a workload."""
    W = weights(cfg.qtype, cfg.od, cfg.id, cfg.seed)
    X = activations(cfg.nt, cfg.id, cfg.seed, cfg.sigma, cfg.outlier_p, cfg.outlier_scale)
    return W, X
