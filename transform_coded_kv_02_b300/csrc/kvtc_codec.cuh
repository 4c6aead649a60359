// Per-token codec on the device: quantiser and record packer (encode side), record unpacker (decode side).
//
// Records [NOVA-KV, third abstract of the "SPHERICAL KV" page: "a fixed per-token bit count", fixed-width
// layout]; z/s word = fp16 zero point z | fp16 scale s << 16.
//  keys   (one token, r_words words): word 0 = z/s; storage channels (2k, 2k+1) share slot k: code word
//         1 + u_k, channel 2k at bits [r_k, r_k + b_2k), channel 2k+1 at bits [16 + r_k, 16 + r_k + b_2k+1).
//  values (two tokens 2p, 2p+1, 2 r_words words): words 0 and 1 = their z/s words; channel j has slot j:
//         code word 2 + u_j, token 2p at bits [r_j, r_j + b_j), token 2p+1 at bits [16 + r_j, 16 + r_j + b_j).
// Slots are placed first-fit by the host; a token of a value record owns one 16-bit half of every code word,
// so the two tokens of a record are written independently with 16-bit stores.
//
// Quantiser, one fixed fp32 op sequence (explicit _rn intrinsics, nothing fused), channels with b_j > 0:
//   y'_j = (y_j - mu_j) * inv_sigma_j;  m = min y', M = max y';  z = fp16_rn(sat(m + 0)),
//   s = fp16_rn(sat(M - z));  c_j = clamp(floor(((y'_j - z) / s) * 2^b_j), 0, 2^b_j - 1), all 0 if s == 0.
#pragma once
#include "kvtc_internal.h"
#include "kvtc_ptx.cuh"

namespace kvtc {

__device__ __forceinline__ __half half_sat_rn(float x) {
  return __float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f));
}

__device__ __forceinline__ uint32_t quantize_code(float yp, float zf, float sf, int b) {
  const float t = __fdiv_rn(__fsub_rn(yp, zf), sf);
  const float u = __fmul_rn(t, exp2i(b));
  const float f = fminf(fmaxf(floorf(u), 0.f), (float)((1 << b) - 1));
  return (uint32_t)f;
}

// Warp-per-token quantise + pack. Lane l holds rotated coefficients y[0..3] of storage channels 4l..4l+3.
// rec_s: per-warp shared scratch of >= 2 r_words words. out: the token's record (keys) or the two-token record
// that holds it (values, tokens = true, half = which of the two), or nullptr.
__device__ __forceinline__ void quantize_pack_warp(const TensorDev& td, int set, const float (&y)[4], int lane,
                                                   uint32_t* rec_s, uint32_t* out, bool tokens, int half) {
  const int j0 = 4 * lane;
  const size_t so = (size_t)set * D + j0;
  const uint32_t w4 = *reinterpret_cast<const uint32_t*>(td.widths + so);
  const float4 mu = *reinterpret_cast<const float4*>(td.mu + so);
  const float4 inv = *reinterpret_cast<const float4*>(td.inv_sigma + so);
  const int b[4] = {(int)(w4 & 255u), (int)((w4 >> 8) & 255u), (int)((w4 >> 16) & 255u), (int)(w4 >> 24)};
  const float muv[4] = {mu.x, mu.y, mu.z, mu.w};
  const float invv[4] = {inv.x, inv.y, inv.z, inv.w};
  float yp[4];
  float m = INFINITY, M = -INFINITY;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    yp[i] = __fmul_rn(__fsub_rn(y[i], muv[i]), invv[i]);
    if (b[i] > 0) {
      m = fminf(m, yp[i]);
      M = fmaxf(M, yp[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  }
  __half zh = __ushort_as_half(0), sh = __ushort_as_half(0);
  if (td.nz[set] > 0) {
    zh = half_sat_rn(__fadd_rn(m, 0.f));
    sh = half_sat_rn(__fsub_rn(M, __half2float(zh)));
  }
  const float zf = __half2float(zh), sf = __half2float(sh);
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  if (sf != 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (b[i] > 0) c[i] = quantize_code(yp[i], zf, sf, b[i]);
  }
  const int R = td.r_words;
  const int W = tokens ? 2 * R : R;
  for (int i = lane; i < W; i += 32) rec_s[i] = 0u;
  __syncwarp();
  const uint32_t* sl = td.slots + (size_t)set * D;
  if (!tokens) {  // key slots 2 lane, 2 lane + 1: channel pairs (4l, 4l+1), (4l+2, 4l+3)
    const uint2 sd = *reinterpret_cast<const uint2*>(sl + 2 * lane);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t desc = i ? sd.y : sd.x;
      if (desc) {
        const uint32_t u = desc & 255u, r = (desc >> 8) & 255u;
        atomicOr(&rec_s[1 + u], (c[2 * i] << r) | (c[2 * i + 1] << (16 + r)));
      }
    }
  } else {        // value slots 4l .. 4l+3: this token's code in the low 16 bits of the staged code word
    const uint4 sd = *reinterpret_cast<const uint4*>(sl + 4 * lane);
    const uint32_t dv[4] = {sd.x, sd.y, sd.z, sd.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (dv[i]) {
        const uint32_t u = dv[i] & 255u, r = (dv[i] >> 8) & 255u;
        atomicOr(&rec_s[2 + u], c[i] << r);
      }
    }
  }
  __syncwarp();
  const uint32_t zs = (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
  if (out) {
    if (!tokens) {
      if (lane == 0) rec_s[0] = zs;
      __syncwarp();
      for (int i = lane; i < R; i += 32) out[i] = rec_s[i];
    } else {
      if (lane == 0) out[half] = zs;
      uint16_t* out16 = reinterpret_cast<uint16_t*>(out);
      for (int i = 2 + lane; i < W; i += 32) out16[2 * i + half] = (uint16_t)rec_s[i];
    }
  }
  __syncwarp();
}

// Thread-per-token quantise + pack (the layout of a tensor-core accumulator row). gy(j) returns the
// rotated coefficient of storage channel j; it is called twice per channel (min/max pass, code pass).
// emit(w, v) receives the token's words: keys, w = 0 .. r_words-1 (full words); values, w = 0 (its z/s word)
// and w = 2 .. 2 r_words - 1 (its 16-bit half of code word w, in the low bits of v).
template <class GetY, class Emit>
__device__ __forceinline__ void quantize_pack_thread(const TensorDev& td, int set, bool tokens, GetY gy, Emit emit) {
  const int nz = td.nz[set];
  const size_t so = (size_t)set * D;
  const float* mu = td.mu + so;
  const float* inv = td.inv_sigma + so;
  const uint8_t* wd = td.widths + so;
  float m = INFINITY, M = -INFINITY;
  for (int j = 0; j < nz; ++j) {
    if (__ldg(wd + j) == 0) continue;
    const float yp = __fmul_rn(__fsub_rn(gy(j), __ldg(mu + j)), __ldg(inv + j));
    m = fminf(m, yp);
    M = fmaxf(M, yp);
  }
  __half zh = __ushort_as_half(0), sh = __ushort_as_half(0);
  if (nz > 0) {
    zh = half_sat_rn(__fadd_rn(m, 0.f));
    sh = half_sat_rn(__fsub_rn(M, __half2float(zh)));
  }
  const float zf = __half2float(zh), sf = __half2float(sh);
  const int W = tokens ? 2 * td.r_words : td.r_words;
  uint32_t acc[2 * MAX_RW];
  for (int w = 0; w < W; ++w) acc[w] = 0u;
  const uint32_t* sl = td.slots + so;
  if (sf != 0.f) {
    if (!tokens) {
      for (int k = 0; 2 * k < nz; ++k) {
        const uint32_t desc = __ldg(sl + k);
        if (!desc) continue;
        uint32_t c[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int j = 2 * k + i, b = __ldg(wd + j);
          if (b > 0) c[i] = quantize_code(__fmul_rn(__fsub_rn(gy(j), __ldg(mu + j)), __ldg(inv + j)), zf, sf, b);
        }
        const uint32_t u = desc & 255u, r = (desc >> 8) & 255u;
        acc[1 + u] |= (c[0] << r) | (c[1] << (16 + r));
      }
    } else {
      for (int j = 0; j < nz; ++j) {
        const uint32_t desc = __ldg(sl + j);
        const int b = __ldg(wd + j);
        if (!desc || b == 0) continue;
        const uint32_t c = quantize_code(__fmul_rn(__fsub_rn(gy(j), __ldg(mu + j)), __ldg(inv + j)), zf, sf, b);
        acc[2 + (desc & 255u)] |= c << ((desc >> 8) & 255u);
      }
    }
  }
  emit(0, (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16));
  for (int w = tokens ? 2 : 1; w < W; ++w) emit(w, acc[w]);
}

}  // namespace kvtc
