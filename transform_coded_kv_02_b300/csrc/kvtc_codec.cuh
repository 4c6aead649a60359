// Per-token codec on the device: quantiser and record packer (encode side), record unpacker (decode side).
//
// Record of one token and tensor [NOVA-KV, third abstract of the "SPHERICAL KV" page: "a fixed per-token
// bit count"]: r_words 32-bit words; word 0 = fp16 zero point z | fp16 scale s << 16; channel codes
// LSB-first from bit 0 of word 1 in storage order (widths non-increasing, zero-width channels last).
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
  const int nbits = b[0] + b[1] + b[2] + b[3];
  if (nbits > 0) {
    const uint64_t chunk = (uint64_t)c[0] | ((uint64_t)c[1] << b[0]) | ((uint64_t)c[2] << (b[0] + b[1])) |
                           ((uint64_t)c[3] << (b[0] + b[1] + b[2]));
    const int o = td.offs[so];
    const uint64_t v = chunk << (o & 31);
    atomicOr(&rec_s[1 + (o >> 5)], (uint32_t)v);
    const uint32_t hi = (uint32_t)(v >> 32);
    if (hi) atomicOr(&rec_s[2 + (o >> 5)], hi);
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
  emit(0, (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16));
  uint64_t buf = 0;
  int nb = 0, w = 1;
  for (int j = 0; j < nz; ++j) {
    const int b = __ldg(wd + j);
    uint32_t c = 0;
    if (sf != 0.f) c = quantize_code(__fmul_rn(__fsub_rn(gy(j), __ldg(mu + j)), __ldg(inv + j)), zf, sf, b);
    buf |= (uint64_t)c << nb;
    nb += b;
    if (nb >= 32) {
      emit(w++, (uint32_t)buf);
      buf >>= 32;
      nb -= 32;
    }
  }
  if (nb > 0) emit(w++, (uint32_t)buf);
  for (; w < td.r_words; ++w) emit(w, 0u);
}

// ------------------------------------------------------------------------------------------------------
// decode-side unpacker: channels 4q..4q+3 of one record -> two fp16 pairs holding (c + 1/2) exactly.
// Codes are OR-ed under the fp16 exponent of 1024 (0x6400: value 1024 + c for c < 1024), then 1023.5 is
// subtracted, which is exact for c < 1024.
// ------------------------------------------------------------------------------------------------------
struct QuadDesc {
  uint32_t wq, sh, s1, s2, s3, m0, m1, m2, m3;
};

__device__ __forceinline__ QuadDesc load_quad(const TensorDev& td, int set, int q) {
  const uint4 a = __ldg(td.quads + ((size_t)set * 32 + q) * 2);
  const uint4 b = __ldg(td.quads + ((size_t)set * 32 + q) * 2 + 1);
  QuadDesc d;
  d.wq = a.x & 255u;
  d.sh = (a.x >> 8) & 255u;
  d.s1 = (a.x >> 16) & 255u;
  d.s2 = a.x >> 24;
  d.m0 = a.y;
  d.m1 = a.z;
  d.s3 = a.w;
  d.m2 = b.x;
  d.m3 = b.y;
  return d;
}

__device__ __forceinline__ uint2 unpack_quad(const uint32_t* rec, const QuadDesc& d) {
  const uint32_t w0 = rec[1 + d.wq], w1 = rec[2 + d.wq];
  const uint32_t x = __funnelshift_r(w0, w1, d.sh);
  const uint32_t h01 = (x & d.m0) | ((x << d.s1) & d.m1) | 0x64006400u;
  const uint32_t y = x >> d.s2;
  const uint32_t h23 = (y & d.m2) | ((y << d.s3) & d.m3) | 0x64006400u;
  const __half2 off = __halves2half2(__ushort_as_half(0x63FF), __ushort_as_half(0x63FF));  // 1023.5
  const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&h01), off);
  const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&h23), off);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
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
