// Parity and self-test kernels behind the kv_debug_* entry points.
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// parity and self-test kernels
// ======================================================================================================
__global__ void __launch_bounds__(256) debug_qp_warp_kernel(ParamsDev P, int set, int tensor, const float* y,
                                                            long long n, uint32_t* rec) {
  __shared__ uint32_t rec_s[8][2 * MAX_RW + 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * 8 + warp;
  if (t >= n) return;
  const TensorDev& td = P.t[tensor];
  const float4 v = *reinterpret_cast<const float4*>(y + (size_t)t * D + 4 * lane);
  const float yy[4] = {v.x, v.y, v.z, v.w};
  uint32_t* out = tensor == 0 ? rec + (size_t)t * td.r_words : rec + (size_t)(t >> 1) * 2 * td.r_words;
  quantize_pack_warp(td, set, yy, lane, rec_s[warp], out, tensor == 1, (int)(t & 1));
}

__global__ void __launch_bounds__(128) debug_qp_thread_kernel(ParamsDev P, int set, int tensor, const float* y,
                                                              long long n, uint32_t* rec) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const TensorDev& td = P.t[tensor];
  const float* yr = y + (size_t)t * D;
  if (tensor == 0) {
    uint32_t* out = rec + (size_t)t * td.r_words;
    quantize_pack_thread(td, set, false, [&](int j) { return yr[j]; }, [&](int w, uint32_t val) { out[w] = val; });
  } else {
    uint32_t* out = rec + (size_t)(t >> 1) * 2 * td.r_words;
    const int half = (int)(t & 1);
    quantize_pack_thread(td, set, true, [&](int j) { return yr[j]; }, [&](int w, uint32_t val) {
      if (w == 0)
        out[half] = val;
      else
        reinterpret_cast<uint16_t*>(out)[2 * w + half] = (uint16_t)val;
    });
  }
}

// The tensor-core encode's quantiser and packer (tc_stage_channel + tc_quantize_pack_row, the functions
// encode_tc_kernel's epilogue runs) on given fp32 rotated rows: one CTA of four warps per 128 tokens; thread = token
// row, its coefficients stored into its tensor-memory lane by tcgen05.st where the encode's MMA would leave them.
// Records as the other variants: keys [n][R]; values [ceil(n / 2)][2 R], token t in half t & 1, and a missing
// second token's half left as it was.
constexpr int DQ_TC_SMEM = 100 * 1024;  // also keeps at most two CTAs (256 tensor-memory columns) per SM
__global__ void __launch_bounds__(128, 1) debug_qp_tc_kernel(ParamsDev P, int set, int tensor, const float* y,
                                                             long long n, uint32_t* rec) {
  extern __shared__ __align__(16) uint32_t stage[];
  __shared__ __align__(16) float pmi[4 * (D / 2)], ptc[4 * (D / 2)], phh[D];
  __shared__ __align__(16) uint32_t pbits[D];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, row = tid;
  const TensorDev& td = P.t[tensor];
  const int R = td.r_words, PK = R | 1, PV = 2 * R + 1;
  const int words = tensor == 0 ? TC_TILE * PK : (TC_TILE / 2) * PV;
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 128);
    tmem_relinquish();
  }
  tc_stage_channel(td, tensor, set, row, pmi, ptc, phh, pbits);
  for (int i = tid; i < words; i += 128) stage[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = s_tmem + ((uint32_t)(32 * warp) << 16);
  const long long t = (long long)blockIdx.x * TC_TILE + row;
#pragma unroll 1
  for (int cb = 0; cb < D / 16; ++cb) {
    uint32_t v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = t < n ? __float_as_uint(y[(size_t)t * D + 16 * cb + i]) : 0u;
    tmem_st_32x32b_x16(tacc + 16u * cb, v);
  }
  tmem_st_wait();
  const int nz = td.nz[set];
  uint32_t* const r = tensor == 0 ? stage + row * PK : stage + (row >> 1) * PV;
  const uint32_t hsh = tensor == 0 ? 0u : 16u * (uint32_t)(row & 1);
  const uint32_t zs = tc_quantize_pack_row(tacc, (nz + 15) >> 4, nz, pmi, ptc, phh, pbits, smem_u32(r), hsh);
  r[tensor == 0 ? 0 : (row & 1)] = zs;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t < n) {
    if (tensor == 0) {
      for (int w = 0; w < R; ++w) rec[(size_t)t * R + w] = r[w];
    } else {
      uint32_t* out = rec + (size_t)(t >> 1) * 2 * R;
      const int hf = (int)(t & 1);
      out[hf] = r[hf];
      for (int w = 2; w < 2 * R; ++w)
        reinterpret_cast<uint16_t*>(out)[2 * w + hf] = reinterpret_cast<const uint16_t*>(r)[2 * w + hf];
    }
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(s_tmem, 128);
}

kv_status launch_debug_quantize_pack(const ParamsDev& P, int set, int tensor, const float* y, int64_t n,
                                     uint32_t* rec, int variant, cudaStream_t s) {
  if (variant == 0) {
    debug_qp_warp_kernel<<<(unsigned)((n + 7) / 8), 256, 0, s>>>(P, set, tensor, y, n, rec);
  } else if (variant == 1) {
    debug_qp_thread_kernel<<<(unsigned)((n + 127) / 128), 128, 0, s>>>(P, set, tensor, y, n, rec);
  } else {
    static_assert(TC_TILE * (MAX_RW | 1) * 4 <= DQ_TC_SMEM && (TC_TILE / 2) * (2 * MAX_RW + 1) * 4 <= DQ_TC_SMEM,
                  "record staging of one tile");
    ensure_dyn_smem((const void*)debug_qp_tc_kernel, DQ_TC_SMEM);
    debug_qp_tc_kernel<<<(unsigned)((n + TC_TILE - 1) / TC_TILE), 128, DQ_TC_SMEM, s>>>(P, set, tensor, y, n, rec);
  }
  return launch_check("debug quantize/pack");
}

// The decoder's slot extraction (slot_f16x2) over records: one thread per (record, slot); writes integer codes
// [n tokens][128], c = (A - 1) 2^w of each fp16 value A = 1 + c 2^-w. Keys: slot k of token t gives channels
// 2k, 2k+1; values: slot j of record p gives channel j of tokens 2p, 2p+1.
__global__ void __launch_bounds__(128) debug_unpack_kernel(ParamsDev P, int set, int tensor, const uint32_t* rec,
                                                           long long n, uint16_t* codes) {
  const TensorDev& td = P.t[tensor];
  const int R = td.r_words;
  const long long n_rec = tensor == 0 ? n : (n + 1) / 2;
  const int n_slot = tensor == 0 ? D / 2 : D;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_rec * n_slot) return;
  const long long r = idx / n_slot;
  const int k = (int)(idx - r * n_slot);
  const uint32_t desc = td.slots[(size_t)set * D + k];
  const uint32_t u = desc & 255u, b0 = (desc >> 16) & 255u, b1 = desc >> 24, w = b0 > b1 ? b0 : b1;
  uint32_t dd, mm;
  slot_decode_desc(0u, (desc >> 8) & 255u, w, b0, b1, dd, mm);
  const float sc = exp2i((int)w);
  if (tensor == 0) {
    const uint32_t h2 = slot_f16x2(rec[r * R + 1 + u], dd, mm);
    const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
    codes[r * D + 2 * k] = (uint16_t)((__low2float(hv) - 1.f) * sc);
    codes[r * D + 2 * k + 1] = (uint16_t)((__high2float(hv) - 1.f) * sc);
  } else {
    const uint32_t h2 = slot_f16x2(rec[r * 2 * R + 2 + u], dd, mm);
    const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
    codes[(2 * r) * D + k] = (uint16_t)((__low2float(hv) - 1.f) * sc);
    if (2 * r + 1 < n) codes[(2 * r + 1) * D + k] = (uint16_t)((__high2float(hv) - 1.f) * sc);
  }
}

kv_status launch_debug_unpack(const ParamsDev& P, int set, int tensor, const uint32_t* rec, int64_t n,
                              uint16_t* codes, cudaStream_t s) {
  const long long work = (tensor == 0 ? n : (n + 1) / 2) * (long long)(tensor == 0 ? D / 2 : D);
  debug_unpack_kernel<<<(unsigned)((work + 127) / 128), 128, 0, s>>>(P, set, tensor, rec, n, codes);
  return launch_check("debug unpack");
}

__global__ void wait_selftest_kernel(long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait_bounded(smem_u32(&bar), 0u, limit_ns);  // no arrival will ever come
  __syncthreads();
}

kv_status launch_wait_selftest(cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(g_wait_limit_ns);
  return launch_check("wait self-test");
}

}  // namespace kvtc
