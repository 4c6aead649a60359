"""Seeded synthetic K/V/Q inputs shaped like the workloads of the transform-coded KV cache pages.

This module only draws random numbers and arranges them into tensors. It holds none of the codec's
arithmetic (no statistics, transforms, bit allocation, quantisation or attention), so the CPU oracle and
the CUDA path can both be fed from it without sharing any of the method.

Recipe (the pages give none; the workload descriptions fix the shapes and the distribution family):
  * per (layer, sequence, KV head) a random orthogonal basis Q (QR of a Gaussian matrix with the signs of
    R's diagonal folded in: F. Mezzadri, "How to generate random matrices from the classical compact
    groups", Notices AMS 2007);
  * a token is Q . diag(sqrt(0.9^i)) . z with z ~ N(0, I) (Student-t with nu=4, scaled to unit variance,
    for the heavy-tailed key workload);
  * keys get 4 outlier raw channels (the first 4 of a seeded permutation) multiplied by 10; values none;
  * queries use an independent basis per query head and are scaled by sqrt(d) so that logits have a
    standard deviation of about 1-2 and the softmax is not flat;
  * optionally a rotary position embedding on keys (half-split pairs (i, i+d/2), base 500000);
  * means are zero.
Every stream is keyed by numpy.random.SeedSequence([seed, layer, seq, head, tensor]).
"""
from __future__ import annotations

import dataclasses

import numpy as np

# stream ids (the last SeedSequence key)
_S_KBASIS, _S_VBASIS, _S_QBASIS, _S_OUTLIER = 1, 2, 3, 4
_S_KTOK, _S_VTOK, _S_QTOK, _S_KCAL, _S_VCAL, _S_QCAL = 10, 11, 12, 13, 14, 15


def rng_for(seed: int, layer: int, seq: int, head: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, layer, seq, head, stream]))


def random_orthogonal(d: int, rng: np.random.Generator) -> np.ndarray:
    """Haar-distributed orthogonal d x d matrix (Mezzadri 2007)."""
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))[None, :]


def latent(n: int, d: int, rng: np.random.Generator, dist: str = "gauss", nu: float = 4.0) -> np.ndarray:
    if dist == "gauss":
        return rng.standard_normal((n, d))
    if dist == "student_t":
        return rng.standard_t(nu, size=(n, d)) * np.sqrt((nu - 2.0) / nu)
    raise ValueError(dist)


def rope_half_split(x: np.ndarray, positions: np.ndarray, base: float = 500000.0) -> np.ndarray:
    """Rotary embedding on pairs (i, i + d/2) at the given integer positions (data synthesis only)."""
    n, d = x.shape
    half = d // 2
    inv = base ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = positions.astype(np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[:, :half], x[:, half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=1)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hkv: int
    Hq: int
    d: int
    T: int
    dtype: str                  # "fp32" or "bf16"
    bits: tuple                 # budgets in bits/element (a sweep for the batched workload)
    n_calib: int
    calib: str                  # "separate" | "own_prefix"
    rope: bool
    key_dist: str
    steps: int = 1
    layers: int = 1
    seed: int = 0

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hkv=1, Hq=4, d=128, T=1024, dtype="fp32", bits=(2.75,), n_calib=512,
                     calib="separate", rope=False, key_dist="gauss", seed=0),
    "llama_decode_32k": Workload("llama_decode_32k", B=1, Hkv=8, Hq=32, d=128, T=32768, dtype="bf16",
                                 bits=(2.75,), n_calib=2048, calib="separate", rope=True,
                                 key_dist="gauss", steps=256, seed=1),
    "qwen_batched_8k": Workload("qwen_batched_8k", B=16, Hkv=4, Hq=28, d=128, T=8192, dtype="bf16",
                                bits=(2.0, 3.0, 4.0), n_calib=1024, calib="own_prefix", rope=False,
                                key_dist="student_t", seed=2),
    "llama_long_128k": Workload("llama_long_128k", B=1, Hkv=8, Hq=32, d=128, T=131072, dtype="bf16",
                                bits=(1.33,), n_calib=2048, calib="separate", rope=True,
                                key_dist="gauss", seed=3),
    "llama_prefill_32l": Workload("llama_prefill_32l", B=4, Hkv=8, Hq=32, d=128, T=65536, dtype="bf16",
                                  bits=(2.75,), n_calib=4096, calib="own_prefix", rope=True,
                                  key_dist="gauss", layers=32, seed=4),
}


class HeadDist:
    """Distribution of one (layer, seq-or-shared, KV head): key/value bases, outliers, query bases."""

    def __init__(self, seed: int, layer: int, seq: int, head: int, d: int, g: int, key_dist: str,
                 decay: float = 0.9, n_outliers: int = 4, outlier_scale: float = 10.0):
        self.seed, self.layer, self.seq, self.head = seed, layer, seq, head
        self.d, self.g, self.key_dist = d, g, key_dist
        self.sqrt_spec = np.sqrt(decay ** np.arange(d, dtype=np.float64))
        self.k_basis = random_orthogonal(d, rng_for(seed, layer, seq, head, _S_KBASIS))
        self.v_basis = random_orthogonal(d, rng_for(seed, layer, seq, head, _S_VBASIS))
        qr = rng_for(seed, layer, seq, head, _S_QBASIS)
        self.q_bases = [random_orthogonal(d, qr) for _ in range(g)]
        perm = rng_for(seed, layer, seq, head, _S_OUTLIER).permutation(d)
        self.k_scale = np.ones(d)
        self.k_scale[perm[:n_outliers]] = outlier_scale

    def keys(self, n: int, rng: np.random.Generator, positions=None, rope: bool = False) -> np.ndarray:
        z = latent(n, self.d, rng, self.key_dist)
        k = ((z * self.sqrt_spec) @ self.k_basis.T) * self.k_scale
        if rope:
            k = rope_half_split(k, positions if positions is not None else np.arange(n))
        return k

    def values(self, n: int, rng: np.random.Generator) -> np.ndarray:
        z = latent(n, self.d, rng, "gauss")
        return (z * self.sqrt_spec) @ self.v_basis.T

    def queries(self, n: int, rng: np.random.Generator) -> np.ndarray:
        """n vectors for each of the g query heads of this KV head: shape [g, n, d]."""
        out = np.empty((self.g, n, self.d))
        for j, qb in enumerate(self.q_bases):
            z = latent(n, self.d, rng, "gauss")
            out[j] = ((z * self.sqrt_spec) @ qb.T) * np.sqrt(self.d)
        return out


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 data to the workload's storage type; returns float32 (fp32) or uint16 bf16 bits."""
    if dtype == "fp32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        f = np.ascontiguousarray(x, dtype=np.float32)
        u = f.view(np.uint32).astype(np.uint64)
        # round-to-nearest-even on the upper 16 bits (inputs are finite)
        r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
        return r
    raise ValueError(dtype)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class LayerData:
    """One layer's synthetic tensors. k, v: [B, Hkv, T, d]; q: [steps, B, Hq, d] decode queries;
    calibration sets indexed by set id (h, or b*Hkv+h when each sequence calibrates on its own prefix):
    calib_k/calib_v [n, d], calib_q [g*n, d]. Storage-typed arrays: fp32 or bf16 bits (uint16)."""
    k: np.ndarray
    v: np.ndarray
    q: np.ndarray
    calib_k: list
    calib_v: list
    calib_q: list
    per_seq_params: bool


def make_layer(w: Workload, layer: int = 0, T: int | None = None, steps: int | None = None,
               B: int | None = None) -> LayerData:
    """Generate one layer of workload `w` (optionally with a shorter context / fewer steps / batch for
    small test cases with the same recipe)."""
    T = w.T if T is None else T
    steps = w.steps if steps is None else steps
    B = w.B if B is None else B
    d, g = w.d, w.g
    per_seq = w.calib == "own_prefix" and w.name != "llama_prefill_32l"
    k = np.empty((B, w.Hkv, T, d))
    v = np.empty((B, w.Hkv, T, d))
    q = np.empty((steps, B, w.Hq, d))
    ck, cv, cq = [], [], []
    for b in range(B):
        for h in range(w.Hkv):
            dist_seq = b if per_seq else 0
            hd = HeadDist(w.seed, layer, dist_seq, h, d, g, w.key_dist)
            pos = np.arange(T)
            k[b, h] = hd.keys(T, rng_for(w.seed, layer, b, h, _S_KTOK), pos, w.rope)
            v[b, h] = hd.values(T, rng_for(w.seed, layer, b, h, _S_VTOK))
            qq = hd.queries(steps, rng_for(w.seed, layer, b, h, _S_QTOK))  # [g, steps, d]
            q[:, b, h * g:(h + 1) * g] = np.transpose(qq, (1, 0, 2))
    st = w.dtype
    k_st, v_st = round_to(k, st), round_to(v, st)
    k, v = as_float(k_st), as_float(v_st)      # calibration prefixes see the stored values
    n = w.n_calib
    if per_seq:
        for b in range(B):
            for h in range(w.Hkv):
                hd = HeadDist(w.seed, layer, b, h, d, g, w.key_dist)
                ck.append(k[b, h, :min(n, T)].copy())
                cv.append(v[b, h, :min(n, T)].copy())
                qq = hd.queries(min(n, T), rng_for(w.seed, layer, b, h, _S_QCAL))
                cq.append(qq.reshape(-1, d))
    else:
        for h in range(w.Hkv):
            hd = HeadDist(w.seed, layer, 0, h, d, g, w.key_dist)
            if w.calib == "own_prefix":          # slice of sequence 0 shared by the batch
                ck.append(k[0, h, :min(n, T)].copy())
                cv.append(v[0, h, :min(n, T)].copy())
                nn = min(n, T)
            else:                                # separate calibration tokens
                ck.append(hd.keys(n, rng_for(w.seed, layer, 0, h, _S_KCAL), np.arange(n), w.rope))
                cv.append(hd.values(n, rng_for(w.seed, layer, 0, h, _S_VCAL)))
                nn = n
            qq = hd.queries(nn, rng_for(w.seed, layer, 0, h, _S_QCAL))
            cq.append(qq.reshape(-1, d))
    return LayerData(k=k_st, v=v_st, q=round_to(q, "bf16"),
                     calib_k=[np.asarray(x, np.float32) for x in ck],
                     calib_v=[np.asarray(x, np.float32) for x in cv],
                     calib_q=[np.asarray(x, np.float32) for x in cq], per_seq_params=per_seq)


def as_float(x: np.ndarray) -> np.ndarray:
    """Storage-typed array -> float64 values (bf16 bits are widened exactly)."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def torch_seed(seed: int, layer: int, seq: int, head: int, stream: int) -> int:
    """A 63-bit seed for torch's generator, derived from the same stream key as rng_for."""
    s = np.random.SeedSequence([seed, layer, seq, head, stream]).generate_state(1, np.uint64)[0]
    return int(s) & ((1 << 63) - 1)


@dataclasses.dataclass
class DeviceLayerData:
    """One layer drawn on a torch device. k, v: bf16 device tensors [B, Hkv, T, d]; q: bf16 bits [1, B, Hq, d]
    (host); calibration sets as in LayerData (host fp32, the stored values)."""
    k: object
    v: object
    q: np.ndarray
    calib_k: list
    calib_v: list
    calib_q: list
    per_seq_params: bool


def make_layer_device(w: Workload, layer: int, device, T: int | None = None,
                      B: int | None = None) -> DeviceLayerData:
    """Workload `w`'s recipe with the token streams drawn by torch's generator on `device`, for layers too
    large to draw on the host (the prefill stack: 4 x 8 x 65536 tokens per layer, 32 layers). The bases,
    outlier channels, spectra and queries are the host recipe's; the Gaussian latents of keys and values come
    from torch (one generator per stream, seeded by torch_seed) and are mixed in fp32, the rotary angles are
    taken in fp64 on the host. One parameter set per KV head, calibrated on tokens 0 .. n_calib - 1 of
    sequence 0 (the prefix shared by the batch). Gaussian keys only."""
    import torch

    if w.key_dist != "gauss" or w.calib != "own_prefix":
        raise ValueError("device draws cover Gaussian keys with a shared calibration prefix")
    T = w.T if T is None else T
    B = w.B if B is None else B
    d, g = w.d, w.g
    k = torch.empty((B, w.Hkv, T, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((B, w.Hkv, T, d), dtype=torch.bfloat16, device=device)
    q = np.empty((1, B, w.Hq, d))
    if w.rope:
        half = d // 2
        inv = 500000.0 ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
        ang = np.arange(T, dtype=np.float64)[:, None] * inv[None, :]
        cos = torch.from_numpy(np.cos(ang).astype(np.float32)).to(device)
        sin = torch.from_numpy(np.sin(ang).astype(np.float32)).to(device)
    ck, cv, cq = [], [], []
    for h in range(w.Hkv):
        hd = HeadDist(w.seed, layer, 0, h, d, g, w.key_dist)
        spec = torch.from_numpy(hd.sqrt_spec.astype(np.float32)).to(device)
        kb = torch.from_numpy(hd.k_basis.T.astype(np.float32)).to(device)
        vb = torch.from_numpy(hd.v_basis.T.astype(np.float32)).to(device)
        ks = torch.from_numpy(hd.k_scale.astype(np.float32)).to(device)
        for b in range(B):
            gen = torch.Generator(device=device)
            gen.manual_seed(torch_seed(w.seed, layer, b, h, _S_KTOK))
            x = (torch.randn((T, d), generator=gen, device=device) * spec) @ kb * ks
            if w.rope:
                a, c = x[:, :d // 2], x[:, d // 2:]
                x = torch.cat([a * cos - c * sin, a * sin + c * cos], dim=1)
            k[b, h] = x.to(torch.bfloat16)
            gen.manual_seed(torch_seed(w.seed, layer, b, h, _S_VTOK))
            v[b, h] = ((torch.randn((T, d), generator=gen, device=device) * spec) @ vb).to(torch.bfloat16)
            qq = hd.queries(1, rng_for(w.seed, layer, b, h, _S_QTOK))  # [g, 1, d]
            q[0, b, h * g:(h + 1) * g] = qq[:, 0]
        n = min(w.n_calib, T)
        ck.append(k[0, h, :n].float().cpu().numpy())
        cv.append(v[0, h, :n].float().cpu().numpy())
        cq.append(np.asarray(hd.queries(n, rng_for(w.seed, layer, 0, h, _S_QCAL)).reshape(-1, d), np.float32))
    return DeviceLayerData(k=k, v=v, q=round_to(q, "bf16"), calib_k=ck, calib_v=cv, calib_q=cq,
                           per_seq_params=False)
