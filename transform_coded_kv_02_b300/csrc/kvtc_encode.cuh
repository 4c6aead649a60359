// Encode, warp per token: rotation on CUDA cores, then the warp quantiser/packer.
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// encode: warp per token
// ======================================================================================================
struct EncArgs {
  const void* src[2];  // [Z][Hkv][t_new][D]
  CacheView c;
  const int64_t* dst_pos;  // [B]: write position of each sequence's first new token (every layer alike)
  int Z;                   // virtual sequences (layers x sequences)
  long long t_new;
  long long wait_ns;
};

template <bool BF16>
__global__ void __launch_bounds__(256) encode_warp_kernel(ParamsDev P, EncArgs a) {
  __shared__ uint32_t rec_s[8][2 * MAX_RW + 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = a.c.Hkv;
  const long long per_tensor = (long long)a.Z * Hkv * a.t_new;
  const long long idx = (long long)blockIdx.x * 8 + warp;
  if (idx >= 2 * per_tensor) return;
  const int tensor = (int)(idx / per_tensor);
  long long r = idx - (long long)tensor * per_tensor;
  const long long t = r % a.t_new;
  r /= a.t_new;
  const int h = (int)(r % Hkv);
  const int z = (int)(r / Hkv);
  const int set = view_set(a.c, z, h);
  const TensorDev& td = P.t[tensor];
  const size_t xo = (((size_t)z * Hkv + h) * a.t_new + t) * D + 4 * lane;
  float x[4];
  if (BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.src[tensor]) + xo);
    x[0] = bf16_bits_f(u.x & 0xFFFFu);
    x[1] = bf16_bits_f(u.x >> 16);
    x[2] = bf16_bits_f(u.y & 0xFFFFu);
    x[3] = bf16_bits_f(u.y >> 16);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(a.src[tensor]) + xo);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  }
  // y_j = sum_k T[j][k] x_k for j = 4 lane + i, reading row k of T^T (coalesced float4 per lane)
  const float4* TT = reinterpret_cast<const float4*>(td.TT + (size_t)set * D * D) + lane;
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int k4 = 0; k4 < 32; ++k4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float xk = __shfl_sync(0xffffffffu, x[i], k4);
      const float4 tt = __ldg(TT + (size_t)(4 * k4 + i) * 32);
      y[0] = fmaf(tt.x, xk, y[0]);
      y[1] = fmaf(tt.y, xk, y[1]);
      y[2] = fmaf(tt.z, xk, y[2]);
      y[3] = fmaf(tt.w, xk, y[3]);
    }
  }
  const long long pos = a.dst_pos[z % a.c.B] + t;
  uint32_t* out = nullptr;
  if (pos >= 0 && pos < a.c.T_cap)
    out = tensor == 0 ? view_key_record(a.c, z, h, pos, td.r_words) : view_value_record(a.c, z, h, pos, td.r_words);
  if (!out && lane == 0) atomicOr(&g_status, ST_BAD_INDEX);
  quantize_pack_warp(td, set, y, lane, rec_s[warp], out, tensor == 1, (int)(pos & 1));
}

// ---- append: one CTA per (tensor, sequence, KV head), its few new tokens one after another ---------------
// T^T arrives in shared memory by one bulk copy while every thread fetches its channel's parameters and the write
// position (one round of loads). Thread j then forms y_j = sum_k T[j][k] x_k with the same FMA chain, in the same k
// order, as encode_warp_kernel, and quantises channel j with the same op sequence as the warp quantiser, so both
// kernels write identical records; the block reduces min and max over the coded channels, and the codes meet in
// the record by shared-memory ORs. One launch costs one transform fetch per head instead of one per token.
constexpr int AP_THREADS = 128;
constexpr int AP_MAX_TOKENS = 16;  // larger appends go to the token-parallel kernels
static size_t append_smem_bytes() { return (size_t)D * D * 4 + 2 * D * 4; }
static_assert(AP_THREADS == D, "one thread per channel");

template <bool BF16>
__global__ void __launch_bounds__(AP_THREADS) encode_append_kernel(ParamsDev P, EncArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* TTs = reinterpret_cast<float*>(smem);  // [k][j]
  float* xs = TTs + D * D;
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red_m[AP_THREADS / 32], red_M[AP_THREADS / 32];
  __shared__ uint32_t rec_s[2 * MAX_RW + 4];
  // a decode call that follows may start preparing (it waits for this grid before it reads q or any record)
  pdl_launch_dependents();
  const int tensor = blockIdx.y, bh = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, j = tid;
  const int z = bh / a.c.Hkv, h = bh - z * a.c.Hkv;
  const int set = view_set(a.c, z, h);
  const TensorDev& td = tensor == 0 ? P.t[0] : P.t[1];
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(smem_u32(&bar), D * D * 4);
    bulk_g2s(smem_u32(TTs), td.TT + (size_t)set * D * D, D * D * 4, smem_u32(&bar));
  }
  // channel j's parameters and its code's place in the record; the first token's element j; the write position
  const size_t so = (size_t)set * D;
  const float mu = td.mu[so + j], inv = td.inv_sigma[so + j];
  const int bw = td.widths[so + j];
  const int nz = td.nz[set];
  const int R = td.r_words, W = tensor == 0 ? R : 2 * R;
  uint32_t cw = 0, cb = 0;  // code word of the record and bit (values: within this token's 16-bit half)
  if (tensor == 0) {
    const uint32_t dsc = td.slots[so + (j >> 1)];
    cw = 1u + (dsc & 255u);
    cb = ((dsc >> 8) & 255u) + 16u * (uint32_t)(j & 1);
  } else {
    const uint32_t dsc = td.slots[so + j];
    cw = 2u + (dsc & 255u);
    cb = (dsc >> 8) & 255u;
  }
  const long long p0 = a.dst_pos[z % a.c.B];
  const void* src = tensor == 0 ? a.src[0] : a.src[1];
  auto load_x = [&](long long t) {
    const size_t xo = ((size_t)bh * a.t_new + t) * D + j;
    return BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(src)[xo]) : static_cast<const float*>(src)[xo];
  };
  float xn = load_x(0);
  bool ok = mbar_wait_bounded(smem_u32(&bar), 0u, a.wait_ns);
  if (!ok && tid == 0) mbar_wait_bounded(smem_u32(&bar), 0u, a.wait_ns);  // drain before leaving
  if (!__syncthreads_and(ok)) return;
  for (long long t = 0; t < a.t_new; ++t) {
    xs[j] = xn;
    if (t + 1 < a.t_new) xn = load_x(t + 1);
    for (int i = tid; i < W; i += AP_THREADS) rec_s[i] = 0u;
    __syncthreads();
    float acc = 0.f;
#pragma unroll 16
    for (int k = 0; k < D; ++k) acc = fmaf(TTs[k * D + j], xs[k], acc);
    // y'_j = (y_j - mu_j) * (1/sigma_j); z = fp16(min y'), s = fp16(max y' - z) over the coded channels
    const float yp = __fmul_rn(__fsub_rn(acc, mu), inv);
    float m = bw > 0 ? yp : INFINITY, M = bw > 0 ? yp : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    if (lane == 0) {
      red_m[warp] = m;
      red_M[warp] = M;
    }
    __syncthreads();
    m = fminf(fminf(red_m[0], red_m[1]), fminf(red_m[2], red_m[3]));
    M = fmaxf(fmaxf(red_M[0], red_M[1]), fmaxf(red_M[2], red_M[3]));
    __half zh = __ushort_as_half(0), sh = __ushort_as_half(0);
    if (nz > 0) {
      zh = half_sat_rn(__fadd_rn(m, 0.f));
      sh = half_sat_rn(__fsub_rn(M, __half2float(zh)));
    }
    const float zf = __half2float(zh), sf = __half2float(sh);
    if (sf != 0.f && bw > 0) atomicOr(&rec_s[cw], quantize_code(yp, zf, sf, bw) << cb);
    __syncthreads();
    const long long pos = p0 + t;
    const uint32_t zs = (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
    uint32_t* out = nullptr;
    if (pos >= 0 && pos < a.c.T_cap)
      out = tensor == 0 ? view_key_record(a.c, z, h, pos, R) : view_value_record(a.c, z, h, pos, R);
    if (out) {
      if (tensor == 0) {
        for (int i = tid; i < R; i += AP_THREADS) out[i] = i == 0 ? zs : rec_s[i];
      } else {
        // the token's half of its two-token record: its z/s word and its 16-bit half of every code word
        const int hf = (int)(pos & 1);
        for (int i = tid; i < W; i += AP_THREADS) {
          if (i < 2) {
            if (i == hf) out[i] = zs;
          } else {
            reinterpret_cast<uint16_t*>(out)[2 * i + hf] = (uint16_t)rec_s[i];
          }
        }
      }
    } else if (tid == 0) {
      atomicOr(&g_status, ST_BAD_INDEX);
    }
    __syncthreads();
  }
}

// path: 0 = automatic, 1 = CUDA cores (append kernel for a few tokens per head, else warp per token),
// 2 = tensor cores (bf16 only). Every path writes records within the codec's end-to-end bar; the two CUDA-core
// kernels write identical records.
kv_status launch_encode(const ParamsDev& P, const CacheView& c, const void* k, const void* v, int dtype, int Z,
                        int64_t t_new, const int64_t* dst_pos, int path, cudaStream_t s) {
  if (path == 2 && dtype != KV_DTYPE_BF16) {
    set_error("the tensor-core encode takes bf16 tokens only");
    return KV_ERR_UNSUPPORTED;
  }
  if (path == 2 || (path == 0 && dtype == KV_DTYPE_BF16 && t_new >= TC_TILE)) {
    const kv_status st = launch_encode_tc(P, c, k, v, Z, t_new, dst_pos, s);
    if (st != KV_ERR_UNSUPPORTED || path == 2) return st;
    clear_error();
  }
  EncArgs a;
  a.src[0] = k;
  a.src[1] = v;
  a.c = c;
  a.dst_pos = dst_pos;
  a.Z = Z;
  a.t_new = t_new;
  a.wait_ns = g_wait_limit_ns;
  if (t_new <= AP_MAX_TOKENS) {
    const size_t smem = append_smem_bytes();
    const dim3 grid((unsigned)(Z * c.Hkv), 2);
    const void* fn = dtype == KV_DTYPE_BF16 ? (const void*)encode_append_kernel<true>
                                            : (const void*)encode_append_kernel<false>;
    const cudaError_t e = ensure_dyn_smem(fn, smem);
    if (e != cudaSuccess) {
      set_error("encode_append_kernel shared memory: %s", cudaGetErrorString(e));
      return KV_ERR_CUDA;
    }
    if (dtype == KV_DTYPE_BF16)
      encode_append_kernel<true><<<grid, AP_THREADS, smem, s>>>(P, a);
    else
      encode_append_kernel<false><<<grid, AP_THREADS, smem, s>>>(P, a);
    return launch_check("encode_append_kernel");
  }
  const long long warps = 2LL * Z * c.Hkv * t_new;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (dtype == KV_DTYPE_BF16)
    encode_warp_kernel<true><<<blocks, 256, 0, s>>>(P, a);
  else
    encode_warp_kernel<false><<<blocks, 256, 0, s>>>(P, a);
  return launch_check("encode_warp_kernel");
}

}  // namespace kvtc
