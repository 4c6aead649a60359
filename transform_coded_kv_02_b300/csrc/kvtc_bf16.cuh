// Uncompressed bf16 split-K flash-decode (the measurement comparator).
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// uncompressed bf16 split-K flash-decode (comparator)
// ======================================================================================================
// A CTA of eight warps owns one split of one (sequence, KV head). Tiles of 128 tokens of K and V stream through a
// ring of shared-memory stages by tiled TMA (one thread issues four 128-row x 64-channel boxes per tile, 128-byte
// swizzle, completion on the stage's mbarrier), so that ldmatrix reads are free of bank conflicts; one barrier per
// tile. The V rows of a partial last tile past the split's end are zeroed before use (K rows there are masked). Warp w
// takes tokens [16 w, 16 w + 16) of each tile: logits on the MMA (A = the g query rows, B = K), online softmax in
// the accumulator layout, P (bf16 hi + lo) straight into the B operand of the P.V MMA (A = V^T). The splits merge
// through the workspace; the last to arrive writes the output.
constexpr int BT = 128;                  // tokens per tile
constexpr int BWARPS = 8;
constexpr int BTHREADS = 32 * BWARPS;
constexpr int BSTAGES = 3;
constexpr int BROW = D * 2;              // bytes per token row
constexpr int BSTAGE_BYTES = 2 * BT * BROW;

struct DecBf16Args {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  unsigned* cnt;    // [B*Hkv] arrival counters: zero before a call, left at zero after it
  float* part;      // [B*Hkv][splits][8][PSTR]
  float* out;
  long long T_cap;
  int B, Hkv, Hq, g, splits;
  float scale_log2;
  int box_rows;       // rows of a TMA box: 128, or all rows of a smaller cache
  long long wait_ns;
};

static size_t decode_bf16_smem_bytes() { return (size_t)BSTAGES * BSTAGE_BYTES + 1024; }  // + alignment slack

// byte offset of 16-byte chunk c (0..15) of token row r in a tile stored as two TMA boxes (channels 0-63, 64-127)
// of 128 rows x 128 bytes with the 128-byte swizzle (chunk index XOR row mod 8)
__device__ __forceinline__ uint32_t bswz(int r, int c) {
  return (uint32_t)((c >> 3) * (BT * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(BTHREADS, 1)
    decode_bf16_kernel(DecBf16Args a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[BSTAGES];
  __shared__ int s_last, s_abort;
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;  // 1024-byte aligned for the swizzle
  uint8_t* const smem = smem_raw + (ring - smem_u32(smem_raw));
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int bh = b * a.Hkv + kh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int g = a.g;
  if (tid == 0) {
    for (int s = 0; s < BSTAGES; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  pdl_wait();
  const long long L = max(0LL, min((long long)a.seq_lens[b], a.T_cap));
  const long long chunk = ((L + a.splits - 1) / a.splits + 15) / 16 * 16;  // this sequence's tokens over the splits
  const long long t0 = min((long long)split * chunk, L);
  const long long t1 = min(t0 + chunk, L);
  const int ntiles = (int)((t1 - t0 + BT - 1) / BT);
  const int row0 = (int)((long long)bh * a.T_cap + t0);  // tensor-map row of the split's first token

  // tile i into ring slot i % BSTAGES (thread 0): K and V, each as two boxes of 64 channels
  auto issue = [&](int i) {
    const uint32_t base = ring + (uint32_t)(i % BSTAGES) * BSTAGE_BYTES;
    const uint32_t bar = smem_u32(&full[i % BSTAGES]);
    const int r = row0 + i * BT;
    mbar_expect_tx(bar, 4u * (uint32_t)a.box_rows * 128u);
    tma_load_2d(base, &mk, 0, r, bar);
    tma_load_2d(base + BT * 128, &mk, 64, r, bar);
    tma_load_2d(base + BT * BROW, &mv, 0, r, bar);
    tma_load_2d(base + BT * BROW + BT * 128, &mv, 64, r, bar);
  };
  int issued = 0;
  if (tid == 0) {
    tma_prefetch_map(&mk);
    tma_prefetch_map(&mv);
    for (int i = 0; i < BSTAGES - 1 && i < ntiles; ++i) issue(i);
    issued = min(BSTAGES - 1, ntiles);
  }

  // q rows (bf16, exact): A row h = head h (h < g), others zero; 8 k-blocks of 16 channels
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
  // ldmatrix rows: lanes 0-7 tokens 0-7 chunk +0, 8-15 tokens 0-7 chunk +1, 16-23 tokens 8-15 +0, 24-31 +1
  const int lr = 16 * warp + (lane & 7) + ((lane >> 4) << 3), lc = (lane >> 3) & 1;

  for (int i = 0; i < ntiles; ++i) {
    // tile i has landed, and every warp is done with tile i - 1
    const bool ok = mbar_wait_bounded(smem_u32(&full[i % BSTAGES]), (uint32_t)((i / BSTAGES) & 1), a.wait_ns);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) s_abort = 1;
      break;
    }
    if (tid == 0 && i + BSTAGES - 1 < ntiles) {
      fence_proxy_async_smem();  // this slot's generic writes (a zeroed tail) before the copy's
      issue(i + BSTAGES - 1);
      issued = i + BSTAGES;
    }
    const uint32_t ks = ring + (uint32_t)(i % BSTAGES) * BSTAGE_BYTES, vs = ks + BT * BROW;
    const long long tb = t0 + (long long)i * BT;
    if (tb + BT > t1) {  // a partial last tile: V rows past the split's end hold whatever the cache holds there
      const int nv = (int)(t1 - tb);
      for (int idx = tid; idx < (BT - nv) * 16; idx += BTHREADS) {
        const int r = nv + (idx >> 4), c = idx & 15;
        *reinterpret_cast<uint4*>(smem + (vs - ring) + bswz(r, c)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    const long long tw = t0 + (long long)i * BT + 16 * warp;  // this warp's first token
    if (tw >= t1) continue;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      uint32_t r0, r1, r2, r3;
      ldsm_x4(ks + bswz(lr, 2 * kb + lc), r0, r1, r2, r3);
      mma_bf16(acc[0], qa[kb], r0, r1);
      mma_bf16(acc[1], qa[kb], r2, r3);
    }
    const int tl[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
    float lg[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) lg[e] = tw + tl[e] < t1 ? a.scale_log2 * acc[e >> 1][e & 1] : -INFINITY;
    float mt = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    const float cr = (m_run == m_new) ? 1.f : ex2_approx(m_run - m_new);
    float p[4], psum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      p[e] = ex2_approx(lg[e] - m_new);
      psum += p[e];
    }
    l_run = fmaf(l_run, cr, psum);
    m_run = m_new;
    __nv_bfloat16 ph[4], pl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ph[e] = __float2bfloat16_rn(p[e]);
      pl[e] = __float2bfloat16_rn(p[e] - __bfloat162float(ph[e]));
    }
    const uint32_t bh0 = pack_bf162(ph[0], ph[1]), bh1 = pack_bf162(ph[2], ph[3]);
    const uint32_t bl0 = pack_bf162(pl[0], pl[1]), bl1 = pack_bf162(pl[2], pl[3]);
    // accumulator columns 2 tig, 2 tig + 1 = heads 2 tig, 2 tig + 1: their factors live in lanes 8 tig, 8 tig + 4
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
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      uint32_t af[4];
      ldsm_x4_t(vs + bswz(lr, 2 * mb + lc), af[0], af[1], af[2], af[3]);
      mma_bf16(acc_o[mb][0], af, bh0, bh1);
      mma_bf16(acc_o[mb][1], af, bl0, bl1);
    }
  }
  if (tid == 0 && s_abort)  // leave no copy in flight
    for (int i = max(0, issued - BSTAGES); i < issued; ++i)
      mbar_wait_bounded(smem_u32(&full[i % BSTAGES]), (uint32_t)((i / BSTAGES) & 1), a.wait_ns);
  __syncthreads();  // the ring is free: the warps' partials go there
  float* ws = reinterpret_cast<float*>(smem);  // [BWARPS][8][PSTR]
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
    float mw[BWARPS];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < BWARPS; ++w) {
      mw[w] = ws[(w * 8 + h) * PSTR];
      M = fmaxf(M, mw[w]);
    }
    float val = 0.f;
    if (cidx == 0) {
      val = M;
    } else if (cidx == 1 || cidx >= 4) {
#pragma unroll
      for (int w = 0; w < BWARPS; ++w) {
        const float e = (mw[w] == -INFINITY) ? 0.f : ex2_approx(mw[w] - M);
        val = fmaf(e, ws[(w * 8 + h) * PSTR + cidx], val);
      }
    }
    part[idx] = val;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.cnt + bh) : "memory");
    const bool last = old == (unsigned)(a.splits - 1);
    if (last) a.cnt[bh] = 0u;  // every split has arrived: the counter is ready for the next call
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  // the last split: weights e_s = 2^(m_s - max m) per head (warp h, lanes over splits), then o = sum e U / sum e l
  const float* pb = a.part + (size_t)bh * a.splits * 8 * PSTR;
  const int S = a.splits;
  float* esw = reinterpret_cast<float*>(smem);  // [MAX_SPLITS][8], then the denominators [8]
  float* den = esw + MAX_SPLITS * 8;
  if (warp < g) {
    const int h = warp;
    float ms[MAX_SPLITS / 32], ls[MAX_SPLITS / 32];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < MAX_SPLITS / 32; ++r) {
      const int sp = min(lane + 32 * r, S - 1);
      ms[r] = __ldcg(pb + ((size_t)sp * 8 + h) * PSTR);
      ls[r] = __ldcg(pb + ((size_t)sp * 8 + h) * PSTR + 1);
      if (lane + 32 * r >= S) ms[r] = -INFINITY;
      M = fmaxf(M, ms[r]);
    }
    M = warp_max(M);
    float dsum = 0.f;
#pragma unroll
    for (int r = 0; r < MAX_SPLITS / 32; ++r) {
      const int sp = lane + 32 * r;
      const float e = ms[r] == -INFINITY ? 0.f : exp2f(ms[r] - M);
      if (sp < S) esw[sp * 8 + h] = e;
      dsum = fmaf(e, ls[r], dsum);
    }
    dsum = warp_sum(dsum);
    if (lane == 0) den[h] = dsum;
  }
  __syncthreads();
  for (int idx = tid; idx < g * D; idx += BTHREADS) {
    const int h = idx >> 7, k = idx & (D - 1);
    const float* ph = pb + (size_t)h * PSTR + 4 + k;
    float o = 0.f;
    constexpr int SB = 16;
    for (int s0 = 0; s0 < S; s0 += SB) {
      float u[SB];
#pragma unroll
      for (int r = 0; r < SB; ++r) u[r] = __ldcg(ph + (size_t)min(s0 + r, S - 1) * 8 * PSTR);
#pragma unroll
      for (int r = 0; r < SB; ++r)
        if (s0 + r < S) o = fmaf(esw[(s0 + r) * 8 + h], u[r], o);
    }
    const float dh = den[h];
    a.out[((size_t)b * a.Hq + (size_t)kh * g + h) * D + k] = dh > 0.f ? o / dh : 0.f;
  }
}

DecodeLayout decode_bf16_layout(int B, int Hkv, int64_t T_cap, int device) {
  DecodeLayout L{};
  split_plan(B, Hkv, T_cap, device, BT, 1, MAX_SPLITS, &L.splits, &L.chunk);
  const size_t bh = (size_t)B * Hkv;
  size_t o = 0;
  L.off_cnt = o;
  o = align256(o + bh * sizeof(unsigned));
  L.off_part = o;
  o = align256(o + bh * (size_t)L.splits * 8 * PSTR * sizeof(float));
  L.total = o;
  return L;
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
  a.B = B;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.g = Hq / Hkv;
  a.splits = L.splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = g_wait_limit_ns;
  const unsigned long long rows = (unsigned long long)B * Hkv * (unsigned long long)T_cap;
  if (rows + BT >= (1ull << 31)) {
    set_error("decode_bf16: %llu cache rows exceed the tensor maps' 32-bit coordinates", rows);
    return KV_ERR_UNSUPPORTED;
  }
  a.box_rows = (int)std::min<unsigned long long>(BT, rows);
  CUtensorMap maps[2];
  if (!make_bf16_map(&maps[0], k, rows, (unsigned)a.box_rows) || !make_bf16_map(&maps[1], v, rows, (unsigned)a.box_rows)) {
    set_error("decode_bf16: tensor map encoding failed");
    return KV_ERR_CUDA;
  }
  const size_t smem = decode_bf16_smem_bytes();
  cudaError_t e = ensure_dyn_smem((const void*)decode_bf16_kernel, smem);
  if (e != cudaSuccess) {
    set_error("decode_bf16_kernel shared memory: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.splits, Hkv, B);
  cfg.blockDim = dim3(BTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_bf16_kernel, a, maps[0], maps[1]);
  if (e != cudaSuccess) {
    set_error("decode_bf16_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return launch_check("decode_bf16_kernel");
}

}  // namespace kvtc
