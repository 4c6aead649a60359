// Per-token codec on the device: quantiser and record packer (encode side), record unpacker (decode side).
//
// Record of one token and tensor [NOVA-KV, third abstract of the "SPHERICAL KV" page: "a fixed per-token
// bit count", fixed-width layout]: r_words 32-bit words; word 0 = fp16 zero point z | fp16 scale s << 16;
// storage channels (2k, 2k+1) share slot k: code word 1 + u_k, channel 2k at bits [r_k, r_k + b_2k),
// channel 2k+1 at bits [16 + r_k, 16 + r_k + b_2k+1) (slots placed first-fit by the host).
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
// rec_s: per-warp shared scratch of >= r_words words. out: global record (r_words words) or nullptr.
__device__ __forceinline__ void quantize_pack_warp(const TensorDev& td, int set, const float (&y)[4], int lane,
                                                   uint32_t* rec_s, uint32_t* out) {
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
  for (int i = lane; i < R; i += 32) rec_s[i] = 0u;
  __syncwarp();
  // lane holds pairs 2 lane and 2 lane + 1
  const uint2 sd = *reinterpret_cast<const uint2*>(td.slots + (size_t)set * (D / 2) + 2 * lane);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t desc = i ? sd.y : sd.x;
    if (desc) {
      const uint32_t u = desc & 255u, r = (desc >> 8) & 255u;
      atomicOr(&rec_s[1 + u], (c[2 * i] << r) | (c[2 * i + 1] << (16 + r)));
    }
  }
  __syncwarp();
  if (lane == 0) rec_s[0] = (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
  __syncwarp();
  if (out)
    for (int i = lane; i < R; i += 32) out[i] = rec_s[i];
  __syncwarp();
}

// Thread-per-token quantise + pack (the layout of a tensor-core accumulator row). gy(j) returns the
// rotated coefficient of storage channel j; it is called twice per channel (min/max pass, code pass).
template <class GetY, class Emit>
__device__ __forceinline__ void quantize_pack_thread(const TensorDev& td, int set, GetY gy, Emit emit) {
  const int nz = td.nz[set];
  const size_t so = (size_t)set * D;
  const float* mu = td.mu + so;
  const float* inv = td.inv_sigma + so;
  const uint8_t* wd = td.widths + so;
  float m = INFINITY, M = -INFINITY;
  for (int j = 0; j < nz; ++j) {
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
  uint32_t acc[MAX_RW];
  for (int w = 0; w < td.r_words; ++w) acc[w] = 0u;
  acc[0] = (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
  const uint32_t* sl = td.slots + (size_t)set * (D / 2);
  for (int k = 0; 2 * k < nz; ++k) {
    const uint32_t desc = __ldg(sl + k);
    if (!desc || sf == 0.f) continue;
    uint32_t c[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = 2 * k + i, b = __ldg(wd + j);
      if (b > 0) c[i] = quantize_code(__fmul_rn(__fsub_rn(gy(j), __ldg(mu + j)), __ldg(inv + j)), zf, sf, b);
    }
    const uint32_t u = desc & 255u, r = (desc >> 8) & 255u;
    acc[1 + u] |= (c[0] << r) | (c[1] << (16 + r));
  }
  for (int w = 0; w < td.r_words; ++w) emit(w, acc[w]);
}

// ------------------------------------------------------------------------------------------------------
// decode-side unpacker: channels 4q..4q+3 (slots 2q, 2q+1) of one record -> two fp16 pairs holding (c + 1/2)
// exactly. A slot's code word shifted right by the slot's bit leaves channel 2k at bit 0 and channel 2k+1 at
// bit 16; both are masked and OR-ed under the fp16 exponent of 1024 (0x6400: value 1024 + c for c < 1024),
// then 1023.5 is subtracted, which is exact.
// ------------------------------------------------------------------------------------------------------
struct QuadDesc {
  uint32_t w0, r0, m0, w1, r1, m1;
};

__device__ __forceinline__ uint32_t slot_mask(uint32_t desc) {
  const uint32_t b0 = (desc >> 16) & 255u, b1 = desc >> 24;
  return ((1u << b0) - 1u) | (((1u << b1) - 1u) << 16);
}

__device__ __forceinline__ QuadDesc load_quad(const TensorDev& td, int set, int q) {
  const uint2 sd = __ldg(reinterpret_cast<const uint2*>(td.slots + (size_t)set * (D / 2)) + q);
  QuadDesc d;
  d.w0 = sd.x & 255u;
  d.r0 = (sd.x >> 8) & 255u;
  d.m0 = slot_mask(sd.x);
  d.w1 = sd.y & 255u;
  d.r1 = (sd.y >> 8) & 255u;
  d.m1 = slot_mask(sd.y);
  return d;
}

__device__ __forceinline__ uint32_t unpack_pair(uint32_t word, uint32_t r, uint32_t m) {
  const uint32_t h = ((word >> r) & m) | 0x64006400u;
  const __half2 off = __halves2half2(__ushort_as_half(0x63FF), __ushort_as_half(0x63FF));  // 1023.5
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint2 unpack_quad(const uint32_t* rec, const QuadDesc& d) {
  return make_uint2(unpack_pair(rec[1 + d.w0], d.r0, d.m0), unpack_pair(rec[1 + d.w1], d.r1, d.m1));
}

// thread -> (quad, first row, row step) of a cooperative unpack over a tile of records
struct QuadMap {
  int q, r0, rstep;
  bool active;
};
__device__ __forceinline__ QuadMap quad_map(int nq, int tid, int nthreads) {
  const int G = nq <= 4 ? 4 : nq <= 8 ? 8 : nq <= 16 ? 16 : 32;
  QuadMap m;
  m.q = tid & (G - 1);
  m.r0 = tid / G;
  m.rstep = nthreads / G;
  m.active = m.q < nq;
  return m;
}

}  // namespace kvtc
