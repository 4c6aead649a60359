// Uncompressed bf16 split-K flash-decode (the measurement comparator).
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// uncompressed bf16 split-K flash-decode (comparator)
// ======================================================================================================
constexpr int BDT = 64;
constexpr int BTHREADS = 128;
constexpr int BSTAGES = 3;
constexpr int BPITCH = 272;  // bytes per token row in shared memory (256 + 16: conflict-free ldmatrix)

struct DecBf16Args {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  unsigned* cnt;
  float* part;
  float* out;
  long long T_cap;
  long long wait_ns;
  int B, Hkv, Hq, g, splits, chunk;
  float scale_log2;
};

static size_t decode_bf16_smem_bytes() { return (size_t)BSTAGES * 2 * BDT * BPITCH + BSTAGES * 8 + 128; }

__global__ void __launch_bounds__(BTHREADS, 2) decode_bf16_kernel(DecBf16Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int bh = b * a.Hkv + kh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int g = a.g;
  const size_t stage_bytes = (size_t)2 * BDT * BPITCH;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BSTAGES * stage_bytes);
  __shared__ int s_last;

  const long long L = min((long long)a.seq_lens[b], a.T_cap);
  const long long t0 = (long long)split * a.chunk;
  const long long t1 = min(t0 + (long long)a.chunk, L);
  const int ntiles = t1 > t0 ? (int)((t1 - t0 + BDT - 1) / BDT) : 0;
  const __nv_bfloat16* kg = a.k + (size_t)bh * a.T_cap * D;
  const __nv_bfloat16* vg = a.v + (size_t)bh * a.T_cap * D;

  auto issue = [&](int i) {  // warp 0, all lanes
    const int s = i % BSTAGES;
    const long long tb = t0 + (long long)i * BDT;
    const int n = (int)min((long long)BDT, t1 - tb);
    const uint32_t bar = smem_u32(&bars[s]);
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)n * 2 * D * 2);
    __syncwarp();
    const uint32_t dk = smem_u32(smem + s * stage_bytes), dv = dk + BDT * BPITCH;
    for (int r = lane; r < n; r += 32) {
      bulk_g2s(dk + r * BPITCH, kg + (tb + r) * D, D * 2, bar);
      bulk_g2s(dv + r * BPITCH, vg + (tb + r) * D, D * 2, bar);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < BSTAGES; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0)
    for (int i = 0; i < min(BSTAGES, ntiles); ++i) issue(i);

  // q rows (bf16, exact): row h = head h (h < g), others zero; 8 k-blocks of 16 channels
  uint32_t qa[8][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + (size_t)kh * g) * D);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      qa[kb][0] = gid < g ? q32[(gid * D + kb * 16 + 2 * tig) >> 1] : 0u;
      qa[kb][1] = 0u;
      qa[kb][2] = gid < g ? q32[(gid * D + kb * 16 + 8 + 2 * tig) >> 1] : 0u;
      qa[kb][3] = 0u;
    }
  }
  float m_run = -INFINITY, l_run = 0.f;
  float acc_o[8][2][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc_o[mb][nb][e] = 0.f;
  const int lrow = (lane & 7) + ((lane >> 4) << 3);
  const int lcol = ((lane >> 3) & 1) * 16;
  int consumed = 0;
  bool aborted = false;
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % BSTAGES;
    const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), (uint32_t)((i / BSTAGES) & 1), a.wait_ns);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      consumed = i;
      break;
    }
    consumed = i + 1;
    uint8_t* ks = smem + s * stage_bytes;
    uint8_t* vs = ks + BDT * BPITCH;
    const long long tile_t0 = t0 + (long long)i * BDT;
    const int lt = warp * 16;
    const bool warp_live = tile_t0 + lt < t1;
    if (warp_live) {
      // rows of this warp's 16 tokens that were not loaded hold stale bytes: zero the value rows so that
      // P = 0 times them stays 0
      for (int r = 0; r < 16; ++r)
        if (tile_t0 + lt + r >= t1) reinterpret_cast<uint2*>(vs + (lt + r) * BPITCH)[lane] = make_uint2(0u, 0u);
      __syncwarp();
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t ka = smem_u32(ks + (lt + lrow) * BPITCH + lcol);
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(ka + kb * 32, r0, r1, r2, r3);
        mma_bf16(acc[0], qa[kb], r0, r1);
        mma_bf16(acc[1], qa[kb], r2, r3);
      }
      const int tl[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
      float lg[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool valid = tile_t0 + lt + tl[e] < t1;
        lg[e] = valid ? a.scale_log2 * acc[e >> 1][e & 1] : -INFINITY;
      }
      float mt = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float m_new = fmaxf(m_run, mt);
      const float cr = (m_run == m_new) ? 1.f : exp2f(m_run - m_new);
      float p[4], psum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = lg[e] == -INFINITY ? 0.f : exp2f(lg[e] - m_new);
        psum += p[e];
      }
      l_run = l_run * cr + psum;
      m_run = m_new;
      __nv_bfloat16 ph[4], pl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ph[e] = __float2bfloat16_rn(p[e]);
        pl[e] = __float2bfloat16_rn(p[e] - __bfloat162float(ph[e]));
      }
      const uint32_t bh0 = pack_bf162(ph[0], ph[1]), bh1 = pack_bf162(ph[2], ph[3]);
      const uint32_t bl0 = pack_bf162(pl[0], pl[1]), bl1 = pack_bf162(pl[2], pl[3]);
      // accumulator columns 2tig, 2tig+1 = heads 2tig, 2tig+1; their maxima live at lanes 8tig, 8tig+4
      const float c_lo = __shfl_sync(0xffffffffu, cr, 8 * tig);
      const float c_hi = __shfl_sync(0xffffffffu, cr, 8 * tig + 4);
      if (__any_sync(0xffffffffu, c_lo != 1.f || c_hi != 1.f)) {
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            acc_o[mb][nb][0] *= c_lo;
            acc_o[mb][nb][1] *= c_hi;
            acc_o[mb][nb][2] *= c_lo;
            acc_o[mb][nb][3] *= c_hi;
          }
      }
      const uint32_t va = smem_u32(vs + (lt + lrow) * BPITCH + lcol);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        uint32_t af[4];
        ldsm_x4_t(va + mb * 32, af[0], af[1], af[2], af[3]);
        mma_bf16(acc_o[mb][0], af, bh0, bh1);
        mma_bf16(acc_o[mb][1], af, bl0, bl1);
      }
    }
    __syncthreads();  // every warp is done with stage s before it is refilled
    if (warp == 0 && i + BSTAGES < ntiles) {
      if (lane == 0) fence_proxy_async_smem();
      __syncwarp();
      issue(i + BSTAGES);
    }
  }
  if (aborted) {
    if (tid == 0)
      for (int i = consumed; i < min(consumed + BSTAGES, ntiles); ++i)
        mbar_wait_bounded(smem_u32(&bars[i % BSTAGES]), (uint32_t)((i / BSTAGES) & 1), a.wait_ns);
    __syncthreads();
    return;
  }
  __syncthreads();
  float* ws = reinterpret_cast<float*>(smem);  // [4][8][PSTR]
  {
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (tig == 0 && gid < g) {
      ws[(warp * 8 + gid) * PSTR + 0] = m_run;
      ws[(warp * 8 + gid) * PSTR + 1] = l;
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const int h0 = 2 * tig, h1 = 2 * tig + 1;
      if (h0 < g) {
        ws[(warp * 8 + h0) * PSTR + 4 + mb * 16 + gid] = acc_o[mb][0][0] + acc_o[mb][1][0];
        ws[(warp * 8 + h0) * PSTR + 4 + mb * 16 + gid + 8] = acc_o[mb][0][2] + acc_o[mb][1][2];
      }
      if (h1 < g) {
        ws[(warp * 8 + h1) * PSTR + 4 + mb * 16 + gid] = acc_o[mb][0][1] + acc_o[mb][1][1];
        ws[(warp * 8 + h1) * PSTR + 4 + mb * 16 + gid + 8] = acc_o[mb][0][3] + acc_o[mb][1][3];
      }
    }
  }
  __syncthreads();
  float* part = a.part + ((size_t)bh * a.splits + split) * 8 * PSTR;
  for (int idx = tid; idx < g * PSTR; idx += BTHREADS) {
    const int h = idx / PSTR, cidx = idx - h * PSTR;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, ws[(w * 8 + h) * PSTR]);
    float val = 0.f;
    if (cidx == 0) {
      val = M;
    } else if (cidx == 1 || cidx >= 4) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = ws[(w * 8 + h) * PSTR];
        const float e = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        val += e * ws[(w * 8 + h) * PSTR + cidx];
      }
    }
    part[idx] = val;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.cnt[bh], 1u) == (unsigned)(a.splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pb = a.part + (size_t)bh * a.splits * 8 * PSTR;
  const int k = tid;
  for (int h = 0; h < g; ++h) {
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; ++sp) M = fmaxf(M, __ldcg(pb + ((size_t)sp * 8 + h) * PSTR));
    float Ls = 0.f, As = 0.f;
    for (int sp = 0; sp < a.splits; ++sp) {
      const float* pp = pb + ((size_t)sp * 8 + h) * PSTR;
      const float ms = __ldcg(pp);
      const float e = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      Ls += e * __ldcg(pp + 1);
      As += e * __ldcg(pp + 4 + k);
    }
    a.out[((size_t)b * a.Hq + (size_t)kh * g + h) * D + k] = Ls > 0.f ? As / Ls : 0.f;
  }
  if (tid == 0) a.cnt[bh] = 0u;
}

DecodeLayout decode_bf16_layout(int B, int Hkv, int64_t T_cap, int device) {
  DecodeLayout L{};
  split_plan(B, Hkv, T_cap, device, BDT, 2, 1 << 20, &L.splits, &L.chunk);
  const size_t bh = (size_t)B * Hkv;
  size_t o = 0;
  L.off_cnt = o;
  o = align256(o + bh * sizeof(unsigned));
  L.off_part = o;
  o = align256(o + bh * (size_t)L.splits * 8 * PSTR * sizeof(float));
  L.total = o;
  return L;
}

__global__ void zero_u32_kernel(unsigned* p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0u;
}

kv_status launch_decode_bf16(const void* k, const void* v, int B, int Hkv, int Hq, int64_t T_cap, const void* q,
                             const int32_t* seq_lens, float scale, float* out, void* ws, const DecodeLayout& L,
                             cudaStream_t s) {
  DecBf16Args a;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_lens = seq_lens;
  a.cnt = reinterpret_cast<unsigned*>(w + L.off_cnt);
  a.part = reinterpret_cast<float*>(w + L.off_part);
  a.out = out;
  a.T_cap = T_cap;
  a.wait_ns = g_wait_limit_ns;
  a.B = B;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.g = Hq / Hkv;
  a.splits = L.splits;
  a.chunk = L.chunk;
  a.scale_log2 = scale * 1.4426950408889634f;
  const int nbh = B * Hkv;
  zero_u32_kernel<<<(nbh + 255) / 256, 256, 0, s>>>(a.cnt, nbh);
  kv_status st = launch_check("zero counters");
  if (st != KV_OK) return st;
  const size_t smem = decode_bf16_smem_bytes();
  const cudaError_t e = ensure_dyn_smem((const void*)decode_bf16_kernel, smem);
  if (e != cudaSuccess) {
    set_error("decode_bf16_kernel shared memory: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  decode_bf16_kernel<<<dim3(L.splits, Hkv, B), BTHREADS, smem, s>>>(a);
  return launch_check("decode_bf16_kernel");
}

}  // namespace kvtc
