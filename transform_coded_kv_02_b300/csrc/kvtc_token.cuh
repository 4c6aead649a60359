// Token-axis allocation on the device: token weights from the attention of observation queries, the tokens each
// (sequence, KV head) keeps, and the compaction of their records. Part of kvtc_kernels.cu's translation unit.
//
// Method: RDKV ("SPHERICAL KV ..." page, first abstract): each token gets a width from full precision down to
// zero bits by reverse water-filling over weights taken from the distortion its compression induces on attention,
// once after the prefill. Here a token's weight is lambda_t = sum_q p_qt^2 over the observation queries q of the
// KV head's query heads (a white error e on token t's value moves query q's output by p_qt e), and the tier above
// zero bits is the token's whole record: reverse water-filling with one tier keeps the `keep` heaviest tokens
// (ties: the earlier token) and evicts the rest. The decode then runs unchanged over the compacted records.
//
//   token_logits_kernel<0|1>  one CTA per run of 128-token tiles of one (sequence, KV head), about two CTAs per
//                             SM: the g x W observation queries (M = 128 rows, zero rows past g W) arrive once by
//                             TMA, the tiles' keys through two stages; a producer warp issues each tile's 8 tcgen05
//                             MMAs (K = 16 each) into one of two 128-column tensor-memory accumulators, so that the
//                             next tile's MMAs and key copy run while this one is read back. Eight epilogue warps,
//                             two on each quarter of the tensor-memory lanes, each thread reading 64 of its lane's
//                             128 logits; mbarriers alone pace them (accumulator done, accumulator released, the
//                             column halves' hand-over), with no CTA-wide barrier per tile.
//                             Pass 0 (lane = query row) leaves each row's maximum and sum of 2^(x - max) over the
//                             run. Pass 1 first merges those runs into each row's M and L (every CTA for its own
//                             sequence and KV head), then takes the transposed product (keys as the MMA's A operand:
//                             lane = token) and sums p^2 = 2^(2 x - 2 (M + log2 L)) over the lane's query columns,
//                             the two halves added through shared memory. The exponentials use the hardware
//                             approximation (relative error about 2^-22), as the decode's softmax does.
//   token_select_kernel       per (sequence, KV head), a cluster of up to 8 CTAs: radix select of the keep-th
//                             largest weight (8 bits per round over the weights' IEEE bits, the CTAs' histograms
//                             summed through distributed shared memory, keys held in shared memory up to 48K tokens
//                             per CTA), then the kept tokens in index order by scans over the CTAs and their warps
//                             (equal weights at the threshold: the earlier tokens).
//   compact_kernel            the kept records copied in order; value tokens re-paired two per record.
#pragma once

#include "kvtc_tc.cuh"

namespace kvtc {

// 32-bit load from a peer CTA's shared memory (an address from dsmem_addr)
__device__ __forceinline__ unsigned ld_dsmem_u32(uint32_t addr) {
  unsigned v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

constexpr int TK_TILE = 128;        // keys per tile and query rows per MMA
constexpr int TK_EPI_WARPS = 8;     // two warps per tensor-memory lane quarter, each over half of the columns
constexpr int TK_THREADS = 32 * (TK_EPI_WARPS + 1);  // and one producer warp (copies and MMAs)
constexpr int SEL_THREADS = 256;  // the selection: one thread per radix digit
static_assert(SEL_THREADS == 256, "the selection kernel gives each thread one 8-bit digit");

struct TokArgs {
  float2* stats;   // [B*Hkv][nch][128]: per run of tiles and query row, (max, sum of 2^(x - max)) over its tokens
  float* lam;      // [B*Hkv][T]:       token weights
  long long T;
  int Hkv, Hq, W, g, nq, nt;
  int tpc, nch;      // tiles per CTA, and the CTAs (runs of tiles) per (sequence, KV head): ceil(nt / tpc)
  int qbox, kbox;    // rows of the query and key boxes: 128, or all rows of a smaller tensor (query rows past qbox
                     // are zeroed in shared memory; key rows past kbox are stale and masked)
  float scale_log2;  // softmax scale * log2(e): logits in base 2
  long long wait_ns;
};

template <int PASS>
__global__ void __launch_bounds__(TK_THREADS, 2)
    token_logits_kernel(TokArgs a, const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk) {
  extern __shared__ uint8_t smem_raw[];
  // by slot (tile parity): keys landed, MMAs done, accumulator released by the eight epilogue warps; pass 1's
  // hand-over of the upper column half's sums, per lane quarter: written, and read
  __shared__ __align__(8) uint64_t qfull, kfull[2], mdone[2], afree[2], pready[2][4], pfree[2][4];
  __shared__ uint32_t s_tmem;
  __shared__ int s_ok;
  __shared__ float cq[TK_TILE];  // pass 1: per query row, 2 (M + log2 L); +inf for rows without a query
  // the upper column half's partial result per lane, by slot: pass 0 (m, l) at the end, pass 1 (sum, -) per tile
  __shared__ float2 part[2][TK_TILE];
  // the queries (two 64-column boxes), then two key stages of two boxes each
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = b * a.Hkv + h;
  const int tile0 = chunk * a.tpc;
  const int ntl = min(a.tpc, a.nt - tile0);  // this CTA's tiles, at least one
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 2 * TK_TILE);
    tmem_relinquish();
  }
  if constexpr (PASS == 1) {  // (M, L) of every query row over pass 0's runs: two threads a row, every other run
    const int row = tid & (TK_TILE - 1), hh = tid >> 7;  // (the producer warp, hh = 2, takes no part)
    const float2* st = a.stats + (size_t)bh * a.nch * TK_TILE + row;
    float mm = -INFINITY, ll = 0.f;
    // eight runs a batch: their loads are independent of one another
    for (int t0 = hh; hh < 2 && t0 < a.nch; t0 += 16) {
      float2 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = t0 + 2 * k < a.nch ? st[(size_t)(t0 + 2 * k) * TK_TILE] : make_float2(-INFINITY, 0.f);
      float mb = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) mb = fmaxf(mb, v[k].x);
      const float mn = fmaxf(mm, mb);
      if (mn != -INFINITY) {
        float lb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) lb += v[k].x == -INFINITY ? 0.f : v[k].y * ex2_approx(v[k].x - mn);
        ll = (mm == -INFINITY ? 0.f : ll * ex2_approx(mm - mn)) + lb;
        mm = mn;
      }
    }
    if (hh == 1) part[0][row] = make_float2(mm, ll);
    __syncthreads();
    if (hh == 0) {
      const float2 o = part[0][row];
      const float M = fmaxf(mm, o.x);
      const float L = M == -INFINITY ? 0.f
                                     : (mm == -INFINITY ? 0.f : ll * ex2_approx(mm - M)) +
                                           (o.x == -INFINITY ? 0.f : o.y * ex2_approx(o.x - M));
      cq[row] = row < a.nq && L > 0.f ? 2.f * (M + log2f(L)) : INFINITY;
    }
  }
  if (a.qbox < TK_TILE) {  // query rows the box does not cover: zeros, so that their logits stay finite
    for (int i = a.qbox * 8 + tid; i < TK_TILE * 8; i += TK_THREADS)
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<uint4*>(smem_raw + (base - smem_u32(smem_raw)) + hf * TC_BOX_BYTES + i * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    mbar_init(smem_u32(&qfull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&kfull[s]), 1);
      mbar_init(smem_u32(&mdone[s]), 1);
      mbar_init(smem_u32(&afree[s]), TK_EPI_WARPS);
      for (int q = 0; q < 4; ++q) {
        mbar_init(smem_u32(&pready[s][q]), 1);
        mbar_init(smem_u32(&pfree[s][q]), 1);
      }
    }
    fence_mbar_init();
    s_ok = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  auto kstage = [&](int s) { return base + (uint32_t)(2 + 2 * s) * TC_BOX_BYTES; };
  // use i of a two-slot barrier: slot i & 1, phase parity (i >> 1) & 1
  auto wait_use = [&](uint64_t& bar, int i) {
    return mbar_wait_bounded(smem_u32(&bar), (uint32_t)(i >> 1) & 1u, a.wait_ns);
  };
  // tensor-memory lane quarter (warp % 4) and column half (warp / 4) of an epilogue warp; r = its lane: pass 0 the
  // query row, pass 1 the tile's token
  const bool epi = warp < TK_EPI_WARPS;
  const int wq = warp & 3, half = warp >> 2;
  const int r = 32 * wq + lane;
  float m = -INFINITY, l = 0.f;  // pass 0: running maximum and sum of 2^(x - max) over this CTA's tokens
  bool all_got = true;
  if (!epi) {
    if (lane == 0) {  // the producer: queries once, keys through the two stages, each tile's MMAs
      int n_load = 0, n_kdone = 0;
      auto load_keys = [&](int i) {  // tile i of this CTA into key stage i & 1 (rows past the head's T are masked)
        const uint32_t fb = smem_u32(&kfull[i & 1]);
        const int krow = (int)((long long)bh * a.T + (long long)(tile0 + i) * TK_TILE);
        mbar_expect_tx(fb, (uint32_t)a.kbox * 256u);
        tma_load_2d(kstage(i & 1), &mk, 0, krow, fb);
        tma_load_2d(kstage(i & 1) + TC_BOX_BYTES, &mk, 64, krow, fb);
        ++n_load;
      };
      const uint32_t qb = smem_u32(&qfull);
      const int qrow = (b * a.Hq + h * a.g) * a.W;  // the g x W observation queries of this KV head
      mbar_expect_tx(qb, (uint32_t)a.qbox * 256u);
      tma_load_2d(base, &mq, 0, qrow, qb);
      tma_load_2d(base + TC_BOX_BYTES, &mq, 64, qrow, qb);
      load_keys(0);
      if (ntl > 1) load_keys(1);
      if (!mbar_wait_bounded(qb, 0u, a.wait_ns)) {
        s_ok = 0;
        mbar_wait_bounded(qb, 0u, a.wait_ns);  // the copy may still land: wait again before the CTA can exit
      }
      for (int i = 0; i < ntl; ++i) {
        const int s = i & 1;
        // accumulator s is free once the epilogue warps are done with tile i - 2; after a failed wait the CTA is
        // marked failed and each remaining tile's barrier is completed without MMAs, so that no warp waits on
        // MMAs that were never issued
        if (i >= 2 && !wait_use(afree[s], i - 2)) s_ok = 0;
        bool issued = false;
        if (s_ok && wait_use(kfull[s], i)) {
          ++n_kdone;
          tc_fence_after();
          constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
          const uint32_t acc = tmem + (uint32_t)(s * TK_TILE);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (uint32_t)(kk >> 2) * TC_BOX_BYTES + (uint32_t)(kk & 3) * 32u;
            // pass 0: logits[query row][token]; pass 1 the transpose, logits[token][query row]
            const uint64_t dq = smem_desc_k128(base + koff), dk = smem_desc_k128(kstage(s) + koff);
            tc_mma_bf16(acc, PASS == 0 ? dq : dk, PASS == 0 ? dk : dq, IDESC, kk ? 1u : 0u);
          }
          tc_commit(smem_u32(&mdone[s]));
          issued = true;
        } else {
          s_ok = 0;
          mbar_arrive(smem_u32(&mdone[s]));
        }
        // the stage takes tile i + 2 once tile i's MMAs have read it
        if (issued && i + 2 < ntl) {
          if (wait_use(mdone[s], i))
            load_keys(i + 2);
          else
            s_ok = 0;
        }
      }
      // before the CTA releases its memory: copies still in flight after a failure, and the last tiles' MMAs (a
      // barrier whose phase has completed, with no later use, passes at once)
      for (int j = n_kdone; j < n_load; ++j) wait_use(kfull[j & 1], j);
      for (int j = max(0, ntl - 2); j < ntl; ++j) wait_use(mdone[j & 1], j);
    }
  } else {
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int cbeg = 64 * half;
    const bool rows_here = PASS == 1 || 32 * wq < a.nq;  // pass 0: warps without a query row read nothing back
    const float two_s = 2.f * a.scale_log2;
    for (int i = 0; i < ntl; ++i) {
      const int s = i & 1;
      const bool got = wait_use(mdone[s], i);
      all_got = all_got && got;
      tc_fence_after();
      const long long t0 = (long long)(tile0 + i) * TK_TILE;
      const int ntok = (int)min((long long)TK_TILE, a.T - t0);
      const uint32_t trow = tmem + lane_off + (uint32_t)(s * TK_TILE);
      if constexpr (PASS == 0) {  // row r's logits (base 2) against the tile's tokens, 32 columns at a time
        for (int c0 = cbeg; c0 < cbeg + 64 && c0 < ntok && rows_here; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(trow + (uint32_t)c0, v);
          tmem_ld_wait();
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]) * a.scale_log2;
          const int nc = min(32, ntok - c0);
          if (nc < 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j >= nc) x[j] = -INFINITY;  // 2^-inf = 0
          }
          // the chunk's maximum as a tree and its sum in four partial sums: short dependency chains
          float t[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) t[j] = fmaxf(x[j], x[j + 16]);
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int j = 0; j < o; ++j) t[j] = fmaxf(t[j], t[j + o]);
          const float mn = fmaxf(m, t[0]);
          float lc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 32; ++j) lc[j & 3] += ex2_approx(x[j] - mn);
          l = (m == -INFINITY ? 0.f : l * ex2_approx(m - mn)) + ((lc[0] + lc[1]) + (lc[2] + lc[3]));
          m = mn;
        }
      } else {  // token r's weight: sum over the query rows of p^2 = 2^(2 s x - 2 (M + log2 L))
        float sum[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: short dependency chains
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c0 = cbeg + 32 * k;
          if (c0 < a.nq) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(trow + (uint32_t)c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[j & 3] += ex2_approx(fmaf(__uint_as_float(v[j]), two_s, -cq[c0 + j]));
          }
        }
        const float sh = (sum[0] + sum[1]) + (sum[2] + sum[3]);
        // the upper half hands its sums to the lower half of the same lane quarter through slot s of part
        if (half) {
          if (i >= 2) wait_use(pfree[s][wq], i - 2);
          part[s][r].x = sh;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&pready[s][wq]));
        } else {
          const bool in = wait_use(pready[s][wq], i);
          const float o = part[s][r].x;
          if (got && in && s_ok && r < ntok) a.lam[(size_t)bh * a.T + t0 + r] = sh + o;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&pfree[s][wq]));
        }
      }
      // this warp is done with accumulator s
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&afree[s]));
    }
  }
  if constexpr (PASS == 0) {  // the two column halves' (m, l) of a row, then the run's statistics
    if (epi && half) part[0][r] = make_float2(m, l);
    __syncthreads();
    if (epi && !half) {
      const float2 o = part[0][r];
      const float mm = fmaxf(m, o.x);
      const float ll = mm == -INFINITY ? 0.f
                                       : (m == -INFINITY ? 0.f : l * ex2_approx(m - mm)) +
                                             (o.x == -INFINITY ? 0.f : o.y * ex2_approx(o.x - mm));
      const bool rv = all_got && s_ok && r < a.nq;
      a.stats[((size_t)bh * a.nch + chunk) * TK_TILE + r] = rv ? make_float2(mm, ll) : make_float2(-INFINITY, 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 2 * TK_TILE);
}

// Exclusive sum over the warps of a per-warp value (every lane of warp w passes the same v): the sum of the warps
// before this one, and the block's total (every thread). Up to 32 warps.
__device__ __forceinline__ unsigned block_warp_excl_sum(unsigned v, unsigned* wsum, unsigned& total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)(blockDim.x >> 5);
  __syncthreads();  // the previous call's readers are done with wsum
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned x = lane < nw ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    wsum[lane] = x;  // inclusive over the warps
  }
  __syncthreads();
  total = wsum[nw - 1];
  return warp ? wsum[warp - 1] : 0u;
}

// Per (sequence, KV head): the keep tokens of largest weight, ascending, found by a cluster of cs CTAs (1, 2, 4 or 8:
// as many as leave every CTA an SM of its own). A weight's rank key is its IEEE bit pattern (monotone for
// non-negative floats); zero, negative and NaN weights rank lowest. CTA c of the cluster owns the token range
// [c Tc, (c + 1) Tc) and its warp w the contiguous sub-range [w C, (w + 1) C), walked 32 tokens at a time (lane =
// token). With KEYS_SMEM the CTA's keys are read from global memory once and kept in dynamic shared memory
// (Tc <= SEL_SMEM_KEYS); otherwise every pass rereads the weights. Radix select, 8 bits a round: each warp counts
// into its own histogram (shared-memory atomics), the CTA sums its warps' histograms per digit, and every CTA sums
// the cluster's CTA histograms through distributed shared memory, so that all of them take the same digit. Output:
// each warp counts its kept tokens (ballots); the CTAs publish their counts above and at the threshold, which gives
// each CTA its first output slot and its share of the keys equal to the threshold (the earliest ones); one exclusive
// sum over the CTA's warps does the same per warp, and each warp writes its tokens in order.
constexpr int SEL_SMEM_KEYS = 48 * 1024;
constexpr int SEL_MAX_CLUSTER = 8;
template <bool KEYS_SMEM>
__global__ void __launch_bounds__(SEL_THREADS, 1)
    token_select_kernel(const float* lam, int T, int keep, int cs, int32_t* idx) {
  extern __shared__ unsigned keys_s[];
  __shared__ unsigned hist[SEL_THREADS / 32][256];
  // this CTA's count per digit, read by the whole cluster; by round parity, so that a round's counts are written
  // while the previous round's may still be read (a peer reads round r's before it arrives at round r + 1's cluster
  // barrier, which every CTA passes before it writes round r + 2's)
  __shared__ unsigned cta_hist[2][256];
  __shared__ unsigned wsum[32];
  __shared__ unsigned s_prefix, s_remaining;
  __shared__ unsigned s_cnt[2];   // this CTA's keys above the threshold and equal to it, read by the later CTAs
  __shared__ unsigned s_base[2];  // keys equal to the threshold and output slots before this CTA
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int crank = (int)cluster_ctarank(), bh = (int)(blockIdx.x / (unsigned)cs);
  const float* lm = lam + (size_t)bh * T;
  int32_t* out = idx + (size_t)bh * keep;
  constexpr int NWS = SEL_THREADS / 32;
  const long long Tc = ((long long)T + cs - 1) / cs;
  const int c0 = (int)min((long long)T, crank * Tc);
  const int n = (int)min((long long)T, c0 + Tc) - c0;                          // this CTA's tokens
  const long long C = (((long long)n + NWS - 1) / NWS + 31) / 32 * 32;         // per warp, whole 32-token chunks
  const int w0 = (int)min((long long)n, warp * C), w1 = (int)min((long long)n, w0 + C);
  auto key_global = [&](int i) {
    const float v = lm[c0 + i];
    return v > 0.f ? __float_as_uint(v) : 0u;
  };
  if constexpr (KEYS_SMEM) {
    for (int i = tid; i < n; i += SEL_THREADS) keys_s[i] = key_global(i);
    __syncthreads();
  }
  auto key_of = [&](int i) {
    if constexpr (KEYS_SMEM) return keys_s[i];
    else return key_global(i);
  };
  // radix select of the keep-th largest key, eight bits per round
  unsigned prefix = 0u, mask = 0u, remaining = (unsigned)keep;
  for (int shift = 24; shift >= 0; shift -= 8) {
    unsigned* const ch = cta_hist[(shift >> 3) & 1];
    for (int i = lane; i < 256; i += 32) hist[warp][i] = 0u;
    __syncwarp();
    for (int b0 = w0; b0 < w1; b0 += 32) {
      const int i = b0 + lane;
      const unsigned k = i < w1 ? key_of(i) : 0u;
      if (i < w1 && (k & mask) == prefix) atomicAdd(&hist[warp][(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 256) {
      unsigned c[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int w = 0; w < NWS; ++w) c[w & 3] += hist[w][tid];
      ch[tid] = (c[0] + c[1]) + (c[2] + c[3]);
    }
    cluster_sync_all();  // every CTA's digit counts are in place
    // digit totals over the cluster, then the count of keys at or above each digit (threads 0..255 take the digits
    // in descending order: an inclusive scan over them); the one digit where the count first reaches `remaining`
    // is the next 8 bits of the threshold
    unsigned dv = 0u, dx = 0u;
    if (tid < 256) {
      const uint32_t a0 = smem_u32(&ch[255 - tid]);
      unsigned pc[SEL_MAX_CLUSTER];  // the cluster's loads issued together
#pragma unroll
      for (int c = 0; c < SEL_MAX_CLUSTER; ++c) pc[c] = c < cs ? ld_dsmem_u32(dsmem_addr(a0, (uint32_t)c)) : 0u;
#pragma unroll
      for (int c = 0; c < SEL_MAX_CLUSTER; ++c) dv += pc[c];
      dx = dv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned nb = __shfl_up_sync(0xffffffffu, dx, o);
        if (lane >= o) dx += nb;
      }
      if (lane == 31) wsum[warp] = dx;
    }
    __syncthreads();
    if (tid < 256) {
      unsigned incl = dx;
      for (int w = 0; w < warp; ++w) incl += wsum[w];
      const unsigned excl = incl - dv;
      if (excl < remaining && remaining <= incl) {
        s_prefix = prefix | ((unsigned)(255 - tid) << shift);
        s_remaining = remaining - excl;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    remaining = s_remaining;
    mask |= 255u << shift;
  }
  // prefix: the threshold key; every larger key is kept, and the first `remaining` keys equal to it
  unsigned n_gt = 0u, n_eq = 0u;
  for (int b0 = w0; b0 < w1; b0 += 32) {
    const int i = b0 + lane;
    const unsigned k = i < w1 ? key_of(i) : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && k > prefix));
    n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && k == prefix));
  }
  unsigned gt_tot, eq_tot;
  const unsigned eq_before_w = block_warp_excl_sum(n_eq, wsum, eq_tot);
  block_warp_excl_sum(n_gt, wsum, gt_tot);
  if (tid == 0) {
    s_cnt[0] = gt_tot;
    s_cnt[1] = eq_tot;
  }
  cluster_sync_all();
  if (tid == 0) {
    unsigned eqb = 0u, slots = 0u;
    for (int c = 0; c < crank; ++c) {
      const unsigned g = ld_dsmem_u32(dsmem_addr(smem_u32(&s_cnt[0]), (uint32_t)c));
      const unsigned e = ld_dsmem_u32(dsmem_addr(smem_u32(&s_cnt[1]), (uint32_t)c));
      slots += g + (eqb >= remaining ? 0u : min(e, remaining - eqb));
      eqb += e;
    }
    s_base[0] = eqb;
    s_base[1] = slots;
  }
  __syncthreads();
  const unsigned eq_before = s_base[0] + eq_before_w;
  const unsigned eq_take = eq_before >= remaining ? 0u : min(n_eq, remaining - eq_before);
  unsigned tot;
  unsigned pos = s_base[1] + block_warp_excl_sum(n_gt + eq_take, wsum, tot);
  unsigned eq_used = 0u;
  const unsigned lt = (1u << lane) - 1u;
  for (int b0 = w0; b0 < w1; b0 += 32) {
    const int i = b0 + lane;
    const unsigned k = i < w1 ? key_of(i) : 0u;
    const bool gt = i < w1 && k > prefix, eq = i < w1 && k == prefix;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_used + __popc(beq & lt) < eq_take);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    const unsigned p = pos + __popc(bsel & lt);
    if (sel && p < (unsigned)keep) out[p] = c0 + i;
    pos += __popc(bsel);
    eq_used += __popc(beq);
  }
  cluster_sync_all();  // the later CTAs have read this CTA's counts before it exits
}

struct CompactArgs {
  const uint32_t* src[2];
  uint32_t* dst[2];
  const int32_t* idx;  // [BH][keep]
  long long Ts, Td;    // token capacities of the source and destination caches
  int keep, Rk, Rv, BH;
};

// keys: thread per (sequence-head, kept token, record word); r = kept token * Rk + word
__device__ __forceinline__ void compact_key_word(const CompactArgs& a, int bh, int r) {
  const int i = r / a.Rk, w = r - i * a.Rk;
  const int t = a.idx[(size_t)bh * a.keep + i];
  if (t < 0 || t >= a.Ts) {
    atomicOr(&g_status, ST_BAD_INDEX);
    return;
  }
  a.dst[0][((size_t)bh * a.Td + i) * a.Rk + w] = a.src[0][((size_t)bh * a.Ts + t) * a.Rk + w];
}

// values: thread per (sequence-head, destination record, record word); kept tokens 2j and 2j + 1 form record j, each
// bringing its z/s word and its 16-bit half of every code word from the record that held it
// r = destination record * 2 Rv + word
__device__ __forceinline__ void compact_value_word(const CompactArgs& a, int bh, int r) {
  const int W = 2 * a.Rv;
  const int j = r / W, w = r - j * W;
  const int32_t* id = a.idx + (size_t)bh * a.keep;
  const int t0 = id[2 * j], t1 = 2 * j + 1 < a.keep ? id[2 * j + 1] : -1;
  if (t0 < 0 || t0 >= a.Ts || (2 * j + 1 < a.keep && (t1 < 0 || t1 >= a.Ts))) {
    atomicOr(&g_status, ST_BAD_INDEX);
    return;
  }
  auto src_word = [&](int t, int word) {
    return a.src[1][((size_t)bh * (a.Ts / 2) + (size_t)(t >> 1)) * W + word];
  };
  uint32_t v;
  if (w < 2) {
    v = w == 0 ? src_word(t0, t0 & 1) : (t1 >= 0 ? src_word(t1, t1 & 1) : 0u);
  } else {
    const uint32_t lo = (src_word(t0, w) >> (16 * (t0 & 1))) & 0xFFFFu;
    const uint32_t hi = t1 >= 0 ? (src_word(t1, w) >> (16 * (t1 & 1))) & 0xFFFFu : 0u;
    v = lo | (hi << 16);
  }
  a.dst[1][((size_t)bh * (a.Td / 2) + (size_t)j) * W + w] = v;
}

// one launch: blockIdx.y = sequence-head, blockIdx.z = 0 for the key words (keep * Rk of them), 1 for the value
// words ((keep + 1) / 2 records of 2 Rv words)
__global__ void compact_kernel(CompactArgs a) {
  const int r = (int)(blockIdx.x * blockDim.x + threadIdx.x), bh = (int)blockIdx.y;
  if (blockIdx.z == 0) {
    if (r < a.keep * a.Rk) compact_key_word(a, bh, r);
  } else if (r < (a.keep + 1) / 2 * 2 * a.Rv) {
    compact_value_word(a, bh, r);
  }
}

// ---- host side --------------------------------------------------------------------------------------------
TokenLayout token_layout(int B, int Hkv, int64_t T) {
  TokenLayout L{};
  L.nt = (int)((T + TK_TILE - 1) / TK_TILE);
  const size_t bh = (size_t)B * Hkv;
  L.off_stats = 0;
  L.total = align256(bh * L.nt * TK_TILE * sizeof(float2));
  return L;
}

kv_status launch_token_weights(const void* q_obs, int W, const void* k, int B, int Hkv, int Hq, int64_t T,
                               float scale, float* lam, void* ws, cudaStream_t s) {
  const TokenLayout L = token_layout(B, Hkv, T);
  CUtensorMap maps[2];
  const unsigned long long qrows = (unsigned long long)B * Hq * W, krows = (unsigned long long)B * Hkv * T;
  const unsigned qbox = (unsigned)std::min<unsigned long long>(128, qrows);
  const unsigned kbox = (unsigned)std::min<unsigned long long>(128, krows);
  if (!make_bf16_map(&maps[0], q_obs, qrows, qbox) || !make_bf16_map(&maps[1], k, krows, kbox)) {
    set_error("token weights: tensor map encoding failed");
    return KV_ERR_CUDA;
  }
  TokArgs a;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.stats = reinterpret_cast<float2*>(w + L.off_stats);
  a.lam = lam;
  a.T = T;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.W = W;
  a.g = Hq / Hkv;
  a.nq = a.g * W;
  a.nt = L.nt;
  // about two CTAs per SM (shared memory admits two), each over a run of tiles of one (sequence, KV head)
  const long long tiles = (long long)L.nt * Hkv * B, target = 2LL * sm_count(current_device());
  a.tpc = (int)std::max(1LL, (tiles + target - 1) / target);
  a.nch = (L.nt + a.tpc - 1) / a.tpc;
  a.qbox = (int)qbox;
  a.kbox = (int)kbox;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = g_wait_limit_ns;
  const uint32_t smem = 1024 + 6 * TC_BOX_BYTES;
  const dim3 grid((unsigned)a.nch, (unsigned)Hkv, (unsigned)B);
  cudaError_t e = ensure_dyn_smem((const void*)token_logits_kernel<0>, smem);
  if (e == cudaSuccess) e = ensure_dyn_smem((const void*)token_logits_kernel<1>, smem);
  if (e != cudaSuccess) {
    set_error("token_logits_kernel shared memory: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  token_logits_kernel<0><<<grid, TK_THREADS, smem, s>>>(a, maps[0], maps[1]);
  token_logits_kernel<1><<<grid, TK_THREADS, smem, s>>>(a, maps[0], maps[1]);
  return launch_check("token weight kernels");
}

kv_status launch_token_select(const float* lam, int B, int Hkv, int64_t T, int64_t keep, int32_t* idx,
                              cudaStream_t s) {
  // one cluster per (sequence, KV head), as many CTAs (of a whole SM each) as the SMs hold for all of them at once
  const long long bh = (long long)B * Hkv;
  const int sms = sm_count(current_device());
  int cs = 1;
  while (cs < SEL_MAX_CLUSTER && bh * cs * 2 <= sms) cs *= 2;
  const long long Tc = (T + cs - 1) / cs;
  const bool in_smem = Tc <= SEL_SMEM_KEYS;
  const size_t smem = in_smem ? (size_t)Tc * 4 : 0;
  if (in_smem) {
    const cudaError_t e = ensure_dyn_smem((const void*)token_select_kernel<true>, smem);
    if (e != cudaSuccess) {
      set_error("token_select_kernel shared memory: %s", cudaGetErrorString(e));
      return KV_ERR_CUDA;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bh * cs), 1, 1);
  cfg.blockDim = dim3(SEL_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = in_smem ? cudaLaunchKernelEx(&cfg, token_select_kernel<true>, lam, (int)T, (int)keep, cs, idx)
                                : cudaLaunchKernelEx(&cfg, token_select_kernel<false>, lam, (int)T, (int)keep, cs, idx);
  if (e != cudaSuccess) {
    set_error("token_select_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return launch_check("token_select_kernel");
}

kv_status launch_compact(const ParamsDev& P, const kv_cache& src, const kv_cache& dst, int B, const int32_t* idx,
                         int64_t keep, cudaStream_t s) {
  CompactArgs a;
  a.src[0] = src.k_rec;
  a.src[1] = src.v_rec;
  a.dst[0] = dst.k_rec;
  a.dst[1] = dst.v_rec;
  a.idx = idx;
  a.Ts = src.T_cap;
  a.Td = dst.T_cap;
  a.keep = (int)keep;
  a.Rk = P.t[0].r_words;
  a.Rv = P.t[1].r_words;
  a.BH = B * src.Hkv;
  const long long per = std::max((long long)keep * a.Rk, (keep + 1) / 2 * 2LL * a.Rv);  // words per head
  if (per == 0) return KV_OK;
  if (per >= (1LL << 31) - 256 || a.BH > 65535) {
    set_error("compaction: %lld record words per head or %d sequence-heads beyond the launch's range", per, a.BH);
    return KV_ERR_UNSUPPORTED;
  }
  compact_kernel<<<dim3((unsigned)((per + 255) / 256), (unsigned)a.BH, 2), 256, 0, s>>>(a);
  return launch_check("compact_kernel");
}

}  // namespace kvtc
