// Encode, warp per token: rotation on CUDA cores, then the warp quantiser/packer.
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// encode: warp per token
// ======================================================================================================
struct EncArgs {
  const void* src[2];
  uint32_t* dst[2];
  const int64_t* dst_pos;
  int B, Hkv, per_seq;
  long long t_new, T_cap;
  long long wait_ns;
};

template <bool BF16>
__global__ void __launch_bounds__(256) encode_warp_kernel(ParamsDev P, EncArgs a) {
  __shared__ uint32_t rec_s[8][2 * MAX_RW + 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long per_tensor = (long long)a.B * a.Hkv * a.t_new;
  const long long idx = (long long)blockIdx.x * 8 + warp;
  if (idx >= 2 * per_tensor) return;
  const int tensor = (int)(idx / per_tensor);
  long long r = idx - (long long)tensor * per_tensor;
  const long long t = r % a.t_new;
  r /= a.t_new;
  const int h = (int)(r % a.Hkv);
  const int b = (int)(r / a.Hkv);
  const int set = a.per_seq ? b * a.Hkv + h : h;
  const TensorDev& td = P.t[tensor];
  const size_t xo = (((size_t)b * a.Hkv + h) * a.t_new + t) * D + 4 * lane;
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
  const long long pos = a.dst_pos[b] + t;
  uint32_t* out = nullptr;
  if (pos >= 0 && pos < a.T_cap) {
    const size_t bh = (size_t)b * a.Hkv + h;
    out = tensor == 0 ? a.dst[0] + (bh * (size_t)a.T_cap + (size_t)pos) * td.r_words
                      : a.dst[1] + (bh * (size_t)(a.T_cap / 2) + (size_t)(pos >> 1)) * 2 * td.r_words;
  } else if (lane == 0) {
    atomicOr(&g_status, ST_BAD_INDEX);
  }
  quantize_pack_warp(td, set, y, lane, rec_s[warp], out, tensor == 1, (int)(pos & 1));
}

// ---- append: one CTA per (tensor, sequence, KV head), its few new tokens one after another ---------------
// T^T arrives in shared memory by one bulk copy; thread j then forms y_j = sum_k T[j][k] x_k with the same FMA
// chain, in the same k order, as encode_warp_kernel, so both kernels write identical records; warp 0 runs the
// warp quantiser/packer. One launch costs one transform fetch per head instead of one per token.
constexpr int AP_THREADS = 128;
constexpr int AP_MAX_TOKENS = 16;  // larger appends go to the token-parallel kernels
static size_t append_smem_bytes() { return (size_t)D * D * 4 + 2 * D * 4; }

template <bool BF16>
__global__ void __launch_bounds__(AP_THREADS) encode_append_kernel(ParamsDev P, EncArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* TTs = reinterpret_cast<float*>(smem);  // [k][j]
  float* xs = TTs + D * D;
  float* ys = xs + D;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t rec_s[2 * MAX_RW + 4];
  // a decode call that follows may start preparing (its q-preparation waits for this grid before it reads q
  // or lets the decode kernel copy records)
  pdl_launch_dependents();
  const int tensor = blockIdx.y, bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int b = bh / a.Hkv, h = bh - b * a.Hkv;
  const int set = a.per_seq ? bh : h;
  const TensorDev& td = P.t[tensor];
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(smem_u32(&bar), D * D * 4);
    bulk_g2s(smem_u32(TTs), td.TT + (size_t)set * D * D, D * D * 4, smem_u32(&bar));
  }
  bool ok = mbar_wait_bounded(smem_u32(&bar), 0u, a.wait_ns);
  if (!ok && tid == 0) mbar_wait_bounded(smem_u32(&bar), 0u, a.wait_ns);  // drain before leaving
  if (!__syncthreads_and(ok)) return;
  for (long long t = 0; t < a.t_new; ++t) {
    const size_t xo = ((size_t)bh * a.t_new + t) * D + tid;
    xs[tid] = BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.src[tensor])[xo])
                   : static_cast<const float*>(a.src[tensor])[xo];
    __syncthreads();
    float acc = 0.f;
#pragma unroll 16
    for (int k = 0; k < D; ++k) acc = fmaf(TTs[k * D + tid], xs[k], acc);
    ys[tid] = acc;
    __syncthreads();
    if (tid < 32) {
      const float4 y4 = reinterpret_cast<const float4*>(ys)[lane];
      const float y[4] = {y4.x, y4.y, y4.z, y4.w};
      const long long pos = a.dst_pos[b] + t;
      uint32_t* out = nullptr;
      if (pos >= 0 && pos < a.T_cap) {
        out = tensor == 0 ? a.dst[0] + ((size_t)bh * a.T_cap + (size_t)pos) * td.r_words
                          : a.dst[1] + ((size_t)bh * (a.T_cap / 2) + (size_t)(pos >> 1)) * 2 * td.r_words;
      } else if (lane == 0) {
        atomicOr(&g_status, ST_BAD_INDEX);
      }
      quantize_pack_warp(td, set, y, lane, rec_s, out, tensor == 1, (int)(pos & 1));
    }
    __syncthreads();
  }
}

// path: 0 = automatic, 1 = CUDA cores (append kernel for a few tokens per head, else warp per token),
// 2 = tensor cores (bf16 only). Every path writes records within the codec's end-to-end bar; the two CUDA-core
// kernels write identical records.
kv_status launch_encode(const ParamsDev& P, const kv_cache& c, const void* k, const void* v, int dtype, int B,
                        int64_t t_new, const int64_t* dst_pos, int path, cudaStream_t s) {
  if (path == 2 && dtype != KV_DTYPE_BF16) {
    set_error("the tensor-core encode takes bf16 tokens only");
    return KV_ERR_UNSUPPORTED;
  }
  if (path == 2 || (path == 0 && dtype == KV_DTYPE_BF16 && t_new >= TC_TILE)) {
    const kv_status st = launch_encode_tc(P, c, k, v, B, t_new, dst_pos, s);
    if (st != KV_ERR_UNSUPPORTED || path == 2) return st;
    clear_error();
  }
  EncArgs a;
  a.src[0] = k;
  a.src[1] = v;
  a.dst[0] = c.k_rec;
  a.dst[1] = c.v_rec;
  a.dst_pos = dst_pos;
  a.B = B;
  a.Hkv = c.Hkv;
  a.per_seq = c.per_seq_params;
  a.t_new = t_new;
  a.T_cap = c.T_cap;
  a.wait_ns = g_wait_limit_ns;
  if (t_new <= AP_MAX_TOKENS) {
    const size_t smem = append_smem_bytes();
    const dim3 grid((unsigned)(B * c.Hkv), 2);
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
  const long long warps = 2LL * B * c.Hkv * t_new;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (dtype == KV_DTYPE_BF16)
    encode_warp_kernel<true><<<blocks, 256, 0, s>>>(P, a);
  else
    encode_warp_kernel<false><<<blocks, 256, 0, s>>>(P, a);
  return launch_check("encode_warp_kernel");
}

}  // namespace kvtc
