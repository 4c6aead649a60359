// Decode over packed records: q preparation and the split-K flash-decode kernel with its launcher.
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
#pragma once

namespace kvtc {

// ======================================================================================================
// decode over packed records
// ======================================================================================================
constexpr int PSTR = 132;          // floats per (split, head) partial: m, l, z, -, A[128]
constexpr int DWARPS = 4;          // token groups per tile: a key warp and a value warp each
constexpr int DT = 16 * DWARPS;    // tokens per ring stage (16 per warp pair)
constexpr int DTHREADS = 64 * DWARPS;  // key warps 0..3, value warps 4..7; lane 0 of warp 0 issues the copies
constexpr int RING_BUDGET = 48 * 1024;
constexpr int MAX_STAGES = 8;
constexpr int MAX_SPLITS = 256;
constexpr int TAIL_RESERVE = MAX_SPLITS * MAX_G * 4 + 4 * MAX_G * 4;  // split weights, head state
static_assert(DTHREADS / 32 >= MAX_G, "one warp per query head of a group in the split merge");

struct DecArgs {
  const uint32_t* rec[2];
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  __half* qa;       // [B*Hkv][16][128]: row 2h (+1) = fp16 hi (lo) part of q' of head h
  float* qc;        // [B*Hkv][QP_PARTS][QPC]: partial C0 of heads 0..7, partial C1 of heads 0..7 (base-2 logits),
                    // the factor 2^-e_h that undoes the scaling of q'_h (the same in every part)
  unsigned* cnt;    // [B*Hkv] arrival counters
  float* part;      // [B*Hkv][splits][g][PSTR] split partials
  float* out;       // [B][Hq][128]
  long long T_cap;
  long long wait_ns;
  int B, Hkv, Hq, g, per_seq, splits, chunk, stages;
  float scale_log2;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- q preparation: QP_PARTS CTAs per (sequence, KV head), 32 rotated channels each ---------------------
constexpr int QPC = 24;  // floats per (sequence, KV head, part) in DecArgs::qc
// q~ = T_K q for the g query heads, read from the transposed transform (T^T row k holds T[j][k] for all j, so the
// 32 lanes of a warp load one coalesced line per k); q'_j = a log2(e) q~_j sigma_j 2^-b_j as fp16 hi + lo;
// partial sums per part of C0 = a log2(e) q.(T_K^T mu) and C1 = a log2(e) sum_{b_j > 0} q~_j sigma_j, which
// the decode kernel adds up. Thread: channel j0 + (tid % 32), k slice 16 (tid / 32) .. + 16.
// q'_h is stored times 2^e_h, e_h = 14 - ceil(log2 B_h) with B_h = |a log2(e)| ||q_h|| max_j sigma_j 2^-b_j >= max_j
// |q'_h,j|: the largest entries then sit near 2^12..2^14, so that the fp16 hi + lo pair keeps about 22 bits for
// every channel that matters instead of sinking into fp16 subnormals when sigma_j 2^-b_j is small; the decode
// multiplies the logit sum by 2^-e_h. Every part computes B_h from the same inputs in the same order.
constexpr int QP_THREADS = 256;
constexpr int QP_PARTS = D / 32;

__global__ void __launch_bounds__(QP_THREADS) qprep_kernel(ParamsDev P, DecArgs a) {
  __shared__ float qs[MAX_G][D];
  __shared__ float red[QP_THREADS / 32][MAX_G][33];
  const int kh = blockIdx.x, b = blockIdx.y, part = blockIdx.z;
  const int bh = b * a.Hkv + kh;
  const int set = a.per_seq ? bh : kh;
  const TensorDev& tk = P.t[0];
  const int g = a.g, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = 32 * part + lane, k0 = 16 * warp;
  // the transform, sigma, widths and the base vector do not depend on earlier kernels: fetch them first
  float t[16];
  const float* TTc = tk.TT + (size_t)set * D * D + j;
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) t[kk] = __ldg(TTc + (size_t)(k0 + kk) * D);
  const float sg = tk.sigma[(size_t)set * D + j];
  const int bw = tk.widths[(size_t)set * D + j];
  const float bk = tk.base[(size_t)set * D + j];
  float sig_step = 0.f;  // max over the nonzero-width channels of sigma_j 2^-b_j (warp 0)
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const int jj = 32 * i + lane;
      const int b2 = tk.widths[(size_t)set * D + jj];
      if (b2 > 0) sig_step = fmaxf(sig_step, tk.sigma[(size_t)set * D + jj] * exp2i(-b2));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sig_step = fmaxf(sig_step, __shfl_xor_sync(0xffffffffu, sig_step, o));
  }
  // This kernel may start while the previous kernel of the stream (an append, say) still runs: wait for it
  // before reading q, and only then release decode_kernel, whose record copies must see every record written
  // before this call.
  pdl_wait();
  pdl_launch_dependents();
  const __nv_bfloat16* qg = a.q + ((size_t)b * a.Hq + (size_t)kh * g) * D;
  for (int i = tid; i < g * D; i += QP_THREADS) qs[i / D][i % D] = __bfloat162float(qg[i]);
  __syncthreads();
#pragma unroll
  for (int h = 0; h < MAX_G; ++h) {
    float acc = 0.f;
    if (h < g) {
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) acc = fmaf(t[kk], qs[h][k0 + kk], acc);
    }
    red[warp][h][lane] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    __half* qa = a.qa + (size_t)bh * 16 * D;
#pragma unroll
    for (int h = 0; h < MAX_G; ++h) {
      float q_t = 0.f;
#pragma unroll
      for (int w = 0; w < QP_THREADS / 32; ++w) q_t += red[w][h][lane];
      float n2 = 0.f;
      if (h < g) {  // warp-uniform
#pragma unroll
        for (int i = 0; i < D / 32; ++i) n2 = fmaf(qs[h][32 * i + lane], qs[h][32 * i + lane], n2);
        n2 = warp_sum(n2);
      }
      const float bound = fabsf(a.scale_log2) * sqrtf(n2) * sig_step;
      int e = 0;
      if (bound > 0.f && bound <= 3.0e38f) {
        int ex;
        frexpf(bound, &ex);  // bound < 2^ex
        e = min(max(14 - ex, -120), 120);
      }
      const bool on = h < g && bw > 0;
      const float qp = on ? a.scale_log2 * q_t * sg * exp2i(-bw) * exp2i(e) : 0.f;
      const __half hi = __float2half_rn(qp);
      const __half lo = __float2half_rn(qp - __half2float(hi));
      qa[(2 * h) * D + j] = hi;
      qa[(2 * h + 1) * D + j] = lo;
      const float c1 = warp_sum(on ? q_t * sg : 0.f);
      if (lane == 0 && h < g) {
        a.qc[(bh * QP_PARTS + part) * QPC + 8 + h] = a.scale_log2 * c1;
        a.qc[(bh * QP_PARTS + part) * QPC + 16 + h] = exp2i(-e);
      }
    }
  } else if (warp == 1) {  // C0 over the query entries k = j0 .. j0 + 31 (the base vector is indexed like q)
#pragma unroll
    for (int h = 0; h < MAX_G; ++h) {
      const float c0 = warp_sum(h < g ? bk * qs[h][j] : 0.f);
      if (lane == 0 && h < g) a.qc[(bh * QP_PARTS + part) * QPC + h] = a.scale_log2 * c0;
    }
  }
  if (tid == 0 && part == 0) a.cnt[bh] = 0u;
}

// ---- split-K decode ----------------------------------------------------------------------------------
constexpr uint32_t PAIR_BYTES_PER_NB = 16u * 8u * 2u + 4u * 4u;  // P tile (16 tokens x 8 columns) + 4 factors

struct DecSmem {  // byte offsets into the dynamic shared memory of decode_kernel
  uint32_t stage_bytes, ps, epi_ws, epi_merged, tail_reserve, total;
};

__host__ __device__ __forceinline__ uint32_t align128u(uint32_t x) { return (x + 127u) & ~127u; }

// main loop: ring | per-pair P tiles and rescale factors
// epilogue (ring dead): T'_V rows [0, 64 KB) | per-warp partials | merged partial
// tail: split partial chunks from 0 | per-split weights and per-head state in the reserve at the end
__host__ __device__ inline DecSmem decode_smem(int RK, int RV, int stages, int nb) {
  DecSmem s;
  s.stage_bytes = (uint32_t)DT * (RK + RV) * 4u;
  s.ps = align128u(stages * s.stage_bytes);
  const uint32_t main_end = s.ps + DWARPS * PAIR_BYTES_PER_NB * nb;
  s.epi_ws = D * D * 4u;
  s.epi_merged = s.epi_ws + DWARPS * 8u * PSTR * 4u;
  const uint32_t epi_end = s.epi_merged + (MAX_G * D + 4 * MAX_G) * 4u;
  s.tail_reserve = align128u(main_end > epi_end ? main_end : epi_end);
  s.total = s.tail_reserve + TAIL_RESERVE;
  return s;
}

__host__ __device__ constexpr int ring_stages_for(int RK, int RV) {
  return (RING_BUDGET / (DT * (RK + RV) * 4)) > MAX_STAGES ? MAX_STAGES
         : (RING_BUDGET / (DT * (RK + RV) * 4)) < 2      ? 2
                                                          : RING_BUDGET / (DT * (RK + RV) * 4);
}

// plain shared-memory word load (byte offset into the dynamic region): the compiler is free to schedule it
template <class T>
__device__ __forceinline__ uint32_t ldsw(const T* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(base) + off);
}

// RT > 0: keys and values both use records of RT words; the ring stage size and count and the offsets between
// a lane's two tokens (two records) are compile-time, so each staged-record address is one add away.
// PIPE: the key warps run the software-pipelined loop (one column block, all eight key channel blocks).
template <int NB, int RT, bool PIPE>
__global__ void __launch_bounds__(DTHREADS, 2) decode_kernel(ParamsDev P, DecArgs a) {
  static_assert(!PIPE || NB == 1, "the pipelined key loop handles one column block");
  extern __shared__ __align__(128) uint8_t smem[];
  // barriers live outside the dynamic region, which the epilogue and the tail reuse wholesale
  __shared__ __align__(8) uint64_t full[MAX_STAGES], empty[MAX_STAGES], pF[DWARPS], pE[DWARPS], tbar_s;
  __shared__ int s_abort, s_last, s_issued;
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int bh = b * a.Hkv + kh;
  const int set = a.per_seq ? bh : kh;
  const TensorDev& TK = P.t[0];
  const TensorDev& TV = P.t[1];
  const int RK = RT ? RT : TK.r_words, RV = RT ? RT : TV.r_words;
  constexpr int NS_CT = RT ? ring_stages_for(RT, RT) : 0;
  const int NS = RT ? NS_CT : a.stages, g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int nzK = TK.nz[set], nzV = TV.nz[set];
  const int nkb = (nzK + 15) >> 4, nmb = (nzV + 15) >> 4;
  const DecSmem L = decode_smem(RK, RV, NS, NB);
  const uint32_t stage_bytes = (uint32_t)DT * (RK + RV) * 4u;
  uint64_t* tbar = &tbar_s;

  // this sequence's tokens spread over all the splits: chunks of whole tiles sized from its own length, so a
  // short sequence in a long cache (or in a ragged batch) keeps every split busy
  const long long Lseq = max(0LL, min((long long)a.seq_lens[b], a.T_cap));
  const long long chunk = ((Lseq + a.splits - 1) / a.splits + DT - 1) / DT * DT;
  const long long t0 = (long long)split * chunk;
  const long long t1 = min(t0 + chunk, Lseq);
  const int ntiles = t1 > t0 ? (int)((t1 - t0 + DT - 1) / DT) : 0;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 2 * DWARPS);  // every key and value warp releases each stage
    }
    for (int p = 0; p < DWARPS; ++p) {
      mbar_init(smem_u32(&pF[p]), 1);
      mbar_init(smem_u32(&pE[p]), 1);
    }
    mbar_init(smem_u32(tbar), 1);
    fence_mbar_init();
    s_abort = 0;
    s_issued = 0;
  }
  __syncthreads();

  // ---- record tiles stream into the ring by bulk copies that lane 0 of warp 0 issues ----
  const uint32_t* krec = a.rec[0] + (size_t)bh * a.T_cap * RK;
  const uint32_t* vrec = a.rec[1] + (size_t)bh * a.T_cap * RV;  // two-token records: same bytes per token
  const bool issuer = tid == 0;
  int next_issue = 0;  // meaningful in the issuing thread only
  auto issue_tile = [&](int i) {
    const int s = i % NS;
    const long long tb = t0 + (long long)i * DT;
    long long n = min((long long)DT, t1 - tb);
    n = min((n + 3) & ~3LL, a.T_cap - tb);
    const uint32_t kbytes = (uint32_t)(n * RK * 4), vbytes = (uint32_t)(n * RV * 4);
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t dst = smem_u32(smem + (size_t)s * stage_bytes);
    mbar_expect_tx(bar, kbytes + vbytes);
    bulk_g2s(dst, krec + tb * RK, kbytes, bar);
    bulk_g2s(dst + DT * RK * 4, vrec + tb * RV, vbytes, bar);
  };
  // issue tiles up to `upto`; blocking: wait for each ring slot to be released, else stop at the first busy one
  auto issue_until = [&](int upto, bool blocking) {
    while (next_issue <= upto && next_issue < ntiles) {
      if (next_issue >= NS) {
        const uint32_t eb = smem_u32(&empty[next_issue % NS]), par = (uint32_t)((next_issue / NS - 1) & 1);
        if (blocking) {
          if (!mbar_wait_bounded(eb, par, a.wait_ns)) {
            s_abort = 1;
            return;
          }
        } else if (!mbar_test(eb, par)) {
          return;
        }
      }
      issue_tile(next_issue);
      ++next_issue;
    }
  };
  if (issuer) {
    if (split == 0 && nzV > 0)  // every split's epilogue reads the scaled T_V rows: warm L2 now
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(TV.Tsc + (size_t)set * D * D),
                   "r"((uint32_t)nzV * D * 4)
                   : "memory");
    issue_until(NS - 1, false);
  }
  // ============ warp pairs: key warp pw and value warp pw + 4 own tokens [16 pw, 16 pw + 16) of every tile ============
  // Codes go from the staged records straight into MMA operand registers.
  //  key warp, logits A operand (16 tokens x 16 channels of block kb): key slot 8kb + tig holds channels
  //    (16kb + 2tig, +1), slot 8kb + 4 + tig channels (16kb + 8 + 2tig, +1); rows gid, gid + 8 = tokens gid, gid + 8.
  //  value warp, P.V A operand (16 channels x 16 tokens): value slot 16mb + gid (+ 8) holds that channel for the
  //    two tokens of a value record; the pair's records tig and tig + 4 hold tokens (2tig, 2tig+1), (2tig+8, 2tig+9).
  // The key warp hands P (fp16 hi/lo of p s_V) and the heads' rescale factors to the value warp through shared
  // memory, guarded by two mbarriers per pair (filled / emptied), whose waits are bounded like every other.
  const int pw = warp & 3;
  const bool kwarp = warp < 4;
  uint8_t* pair_smem = smem + L.ps + (size_t)pw * PAIR_BYTES_PER_NB * NB;
  __half* ps = reinterpret_cast<__half*>(pair_smem);                          // [16 tokens][8 NB columns]
  float* pcorr = reinterpret_cast<float*>(pair_smem + 16 * 8 * NB * 2);       // [NB][4]
  float* ws = reinterpret_cast<float*>(smem + L.epi_ws);                       // [DWARPS][8][PSTR]
  const uint32_t kstep = 8u * RK * 4, vstep = 4u * 2 * RV * 4;
  if (kwarp) {
    const uint32_t krow = (uint32_t)(16 * pw + gid) * RK * 4;
    uint32_t ka[8][2], ks[8][2], km[8][2];
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t dk = kb < nkb ? __ldg(TK.slots + (size_t)set * D + 8 * kb + 4 * i + tig) : 0u;
        ka[kb][i] = krow + 4u * (1u + (dk & 255u));
        ks[kb][i] = (dk >> 8) & 255u;
        km[kb][i] = slot_mask(dk);
      }
    // z/s words: key record of token gid; value record (gid >> 1), half gid & 1; tokens gid + 8 one step on
    const uint32_t kz = krow;
    const uint32_t vz = (uint32_t)DT * RK * 4 + (uint32_t)(8 * pw + (gid >> 1)) * 2 * RV * 4 + 4u * (gid & 1);
    float m_run[NB], l_run[NB], z_run[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      m_run[nb] = -INFINITY;
      l_run[nb] = 0.f;
      z_run[nb] = 0.f;
    }
    // q' (B operand of the logits MMA) and the folded constants come from qprep_kernel
    pdl_wait();
    uint32_t qb[8][NB][2];
    {
      const uint32_t* qa32 = reinterpret_cast<const uint32_t*>(a.qa + (size_t)bh * 16 * D);
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int col = nb * 8 + gid;
          qb[kb][nb][0] = kb < nkb ? qa32[(col * D + kb * 16 + 2 * tig) >> 1] : 0u;
          qb[kb][nb][1] = kb < nkb ? qa32[(col * D + kb * 16 + 8 + 2 * tig) >> 1] : 0u;
        }
    }
    float c0[NB], c1[NB], qsc[NB];  // qsc: 2^-e_h, undoing the scaling of q'
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int h = tig + 4 * nb;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int pt = 0; pt < QP_PARTS; ++pt) {
        s0 += h < g ? a.qc[(bh * QP_PARTS + pt) * QPC + h] : 0.f;
        s1 += h < g ? a.qc[(bh * QP_PARTS + pt) * QPC + 8 + h] : 0.f;
      }
      c0[nb] = s0;
      c1[nb] = s1;
      qsc[nb] = h < g ? a.qc[(size_t)bh * QP_PARTS * QPC + 16 + h] : 0.f;
    }
    int hand = 0;  // handoffs to the value warp so far
    if constexpr (PIPE) {
      // Software pipeline: tile i + 1's record loads, code extraction and logit MMAs are issued in the same
      // straight-line block as tile i's softmax, so that the two interleave. All eight channel blocks are
      // processed (blocks past the last nonzero-width channel hold zero descriptors and meet a zero q').
      const int n_in = (int)(t1 - t0);  // tokens of this split
      float accC[4] = {0.f, 0.f, 0.f, 0.f}, accN[4];
      uint32_t zC[4] = {0u, 0u, 0u, 0u}, zN[4];
      auto tile_logits = [&](int j, float (&acc)[4], uint32_t (&zw)[4]) -> bool {
        const int sj = j % NS;
        const uint8_t* st = smem + (size_t)sj * stage_bytes;
        if (issuer) issue_until(j, true);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[sj]), (uint32_t)((j / NS) & 1), a.wait_ns)))
          return false;
        zw[0] = ldsw(st, kz);
        zw[1] = ldsw(st, kz + kstep);
        zw[2] = ldsw(st, vz);
        zw[3] = ldsw(st, vz + vstep);
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          uint32_t af[4];
          af[0] = unpack_pair(ldsw(st, ka[kb][0]), ks[kb][0], km[kb][0]);
          af[1] = unpack_pair(ldsw(st, ka[kb][0] + kstep), ks[kb][0], km[kb][0]);
          af[2] = unpack_pair(ldsw(st, ka[kb][1]), ks[kb][1], km[kb][1]);
          af[3] = unpack_pair(ldsw(st, ka[kb][1] + kstep), ks[kb][1], km[kb][1]);
          mma_f16(acc, af, qb[kb][0][0], qb[kb][0][1]);
        }
        return true;
      };
      bool ok = ntiles == 0 || tile_logits(0, accC, zC);
      if (!ok) s_abort = 1;
      for (int i = 0; ok && i < ntiles; ++i) {
        // tile i's codes are in registers: release its stage before waiting for the next one
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[i % NS]));
        if (issuer) issue_until(i + NS - 1, false);
        if (i + 1 < ntiles && !tile_logits(i + 1, accN, zN)) {
          s_abort = 1;
          break;
        }
        const int my0 = i * DT + 16 * pw;
        const bool valid0 = my0 + gid < n_in, valid1 = my0 + gid + 8 < n_in;
        // z/s words: fp16 z in the low half, s in the high half
        const float2 zsk0 = __half22float2(*reinterpret_cast<const __half2*>(&zC[0]));
        const float2 zsk1 = __half22float2(*reinterpret_cast<const __half2*>(&zC[1]));
        const float2 zsv0 = __half22float2(*reinterpret_cast<const __half2*>(&zC[2]));
        const float2 zsv1 = __half22float2(*reinterpret_cast<const __half2*>(&zC[3]));
        const float zk0 = zsk0.x, sk0 = zsk0.y, zk1 = zsk1.x, sk1 = zsk1.y;
        const float zv0 = zsv0.x, sv0 = zsv0.y, zv1 = zsv1.x, sv1 = zsv1.y;
        const float r0 = (accC[0] + accC[1]) * qsc[0], r1 = (accC[2] + accC[3]) * qsc[0];
        const float l0 = valid0 ? fmaf(sk0, r0, fmaf(zk0, c1[0], c0[0])) : -INFINITY;
        const float l1 = valid1 ? fmaf(sk1, r1, fmaf(zk1, c1[0], c0[0])) : -INFINITY;
        float mt = fmaxf(l0, l1);
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = fmaxf(m_run[0], mt);
        const float corr = (m_run[0] == m_new) ? 1.f : ex2_approx(m_run[0] - m_new);
        const float p0 = valid0 ? ex2_approx(l0 - m_new) : 0.f;
        const float p1 = valid1 ? ex2_approx(l1 - m_new) : 0.f;
        l_run[0] = fmaf(l_run[0], corr, p0 + p1);
        z_run[0] = fmaf(z_run[0], corr, (valid0 ? p0 * zv0 : 0.f) + (valid1 ? p1 * zv1 : 0.f));
        m_run[0] = m_new;
        const float w0 = valid0 ? p0 * sv0 : 0.f, w1 = valid1 ? p1 * sv1 : 0.f;
        const __half h0 = __float2half_rn(w0), h1 = __float2half_rn(w1);
        const uint32_t e0 = pack_half2(h0, __float2half_rn(w0 - __half2float(h0)));
        const uint32_t e1 = pack_half2(h1, __float2half_rn(w1 - __half2float(h1)));
        if (hand > 0 &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&pE[pw]), (uint32_t)((hand - 1) & 1), a.wait_ns))) {
          s_abort = 1;
          break;
        }
        reinterpret_cast<uint32_t*>(ps)[(gid * 8 + 2 * tig) >> 1] = e0;
        reinterpret_cast<uint32_t*>(ps)[((gid + 8) * 8 + 2 * tig) >> 1] = e1;
        if (gid == 0) pcorr[tig] = corr;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&pF[pw]));
        ++hand;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          accC[e] = accN[e];
          zC[e] = zN[e];
        }
      }
    } else {
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NS;
      const uint8_t* st = smem + (size_t)s * stage_bytes;
      if (issuer) issue_until(i, true);
      // every lane takes the stage's data through its own wait; the verdict is made warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((i / NS) & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
      const long long my_t0 = t0 + (long long)i * DT + 16 * pw;
      if (my_t0 >= t1) {  // this pair's tokens are past the end
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (issuer) issue_until(i + NS - 1, false);
        continue;
      }
      const uint32_t kzw0 = ldsw(st, kz), kzw1 = ldsw(st, kz + kstep);
      const uint32_t vzw0 = ldsw(st, vz), vzw1 = ldsw(st, vz + vstep);
      // ---- logits: A = key codes (16 tokens x 16 channels), B = q' (16 channels x 8 columns) ----
      float acc2[2][NB][4];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc2[u][nb][0] = acc2[u][nb][1] = acc2[u][nb][2] = acc2[u][nb][3] = 0.f;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        if (kb < nkb) {
          uint32_t af[4];
          af[0] = unpack_pair(ldsw(st, ka[kb][0]), ks[kb][0], km[kb][0]);
          af[1] = unpack_pair(ldsw(st, ka[kb][0] + kstep), ks[kb][0], km[kb][0]);
          af[2] = unpack_pair(ldsw(st, ka[kb][1]), ks[kb][1], km[kb][1]);
          af[3] = unpack_pair(ldsw(st, ka[kb][1] + kstep), ks[kb][1], km[kb][1]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16(acc2[kb & 1][nb], af, qb[kb][nb][0], qb[kb][nb][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the key warp is done with the stage
      if (issuer) issue_until(i + NS - 1, false);
      const bool valid0 = my_t0 + gid < t1, valid1 = my_t0 + gid + 8 < t1;
      const float zk0 = half_bits_to_float(kzw0), sk0 = half_bits_to_float(kzw0 >> 16);
      const float zk1 = half_bits_to_float(kzw1), sk1 = half_bits_to_float(kzw1 >> 16);
      const float zv0 = half_bits_to_float(vzw0), sv0 = half_bits_to_float(vzw0 >> 16);
      const float zv1 = half_bits_to_float(vzw1), sv1 = half_bits_to_float(vzw1 >> 16);
      uint32_t e0[NB], e1[NB];
      float corr[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const float r0 = ((acc2[0][nb][0] + acc2[1][nb][0]) + (acc2[0][nb][1] + acc2[1][nb][1])) * qsc[nb];
        const float r1 = ((acc2[0][nb][2] + acc2[1][nb][2]) + (acc2[0][nb][3] + acc2[1][nb][3])) * qsc[nb];
        const float l0 = valid0 ? fmaf(sk0, r0, fmaf(zk0, c1[nb], c0[nb])) : -INFINITY;
        const float l1 = valid1 ? fmaf(sk1, r1, fmaf(zk1, c1[nb], c0[nb])) : -INFINITY;
        float mt = fmaxf(l0, l1);
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = fmaxf(m_run[nb], mt);
        corr[nb] = (m_run[nb] == m_new) ? 1.f : exp2f(m_run[nb] - m_new);
        const float p0 = valid0 ? exp2f(l0 - m_new) : 0.f;
        const float p1 = valid1 ? exp2f(l1 - m_new) : 0.f;
        l_run[nb] = fmaf(l_run[nb], corr[nb], p0 + p1);
        z_run[nb] = fmaf(z_run[nb], corr[nb], (valid0 ? p0 * zv0 : 0.f) + (valid1 ? p1 * zv1 : 0.f));
        m_run[nb] = m_new;
        const float w0 = valid0 ? p0 * sv0 : 0.f, w1 = valid1 ? p1 * sv1 : 0.f;
        const __half h0 = __float2half_rn(w0), h1 = __float2half_rn(w1);
        e0[nb] = pack_half2(h0, __float2half_rn(w0 - __half2float(h0)));
        e1[nb] = pack_half2(h1, __float2half_rn(w1 - __half2float(h1)));
      }
      // ---- hand P and the rescale factors to the value warp ----
      if (hand > 0 &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&pE[pw]), (uint32_t)((hand - 1) & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        reinterpret_cast<uint32_t*>(ps)[(gid * 8 * NB + nb * 8 + 2 * tig) >> 1] = e0[nb];
        reinterpret_cast<uint32_t*>(ps)[((gid + 8) * 8 * NB + nb * 8 + 2 * tig) >> 1] = e1[nb];
        if (gid == 0) pcorr[nb * 4 + tig] = corr[nb];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&pF[pw]));
      ++hand;
    }
    }
    if (issuer) s_issued = next_issue;
    // this pair's softmax state into the per-pair partial (the region lies past the ring)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      l_run[nb] += __shfl_xor_sync(0xffffffffu, l_run[nb], 4);
      l_run[nb] += __shfl_xor_sync(0xffffffffu, l_run[nb], 8);
      l_run[nb] += __shfl_xor_sync(0xffffffffu, l_run[nb], 16);
      z_run[nb] += __shfl_xor_sync(0xffffffffu, z_run[nb], 4);
      z_run[nb] += __shfl_xor_sync(0xffffffffu, z_run[nb], 8);
      z_run[nb] += __shfl_xor_sync(0xffffffffu, z_run[nb], 16);
      const int h = tig + 4 * nb;
      if (h < g && gid == 0) {
        float* w = ws + (pw * 8 + h) * PSTR;
        w[0] = m_run[nb];
        w[1] = l_run[nb];
        w[2] = z_run[nb];
      }
    }
  } else {
    const uint32_t vrow = (uint32_t)DT * RK * 4 + (uint32_t)(8 * pw + tig) * 2 * RV * 4;
    uint32_t va[8][2], vsh[8][2], vm[8][2];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t dv = mb < nmb ? __ldg(TV.slots + (size_t)set * D + 16 * mb + 8 * i + gid) : 0u;
        va[mb][i] = vrow + 4u * (2u + (dv & 255u));
        vsh[mb][i] = (dv >> 8) & 255u;
        vm[mb][i] = slot_mask(dv);
      }
    float acc_o[8][NB][4];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_o[mb][nb][e] = 0.f;
    const uint32_t pa = smem_u32(ps + (lane & 15) * 8 * NB);
    int hand = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NS;
      const uint8_t* st = smem + (size_t)s * stage_bytes;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((i / NS) & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
      const long long my_t0 = t0 + (long long)i * DT + 16 * pw;
      if (my_t0 >= t1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        continue;
      }
      // value codes of this pair's 16 tokens: with one column block they are taken while the key warp works on
      // the logits (and the stage released early); with two, registers are short and they go straight to the MMA
      uint32_t vf[NB == 1 ? 8 : 1][4];
      if constexpr (NB == 1) {
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          if (mb < nmb) {
            vf[mb][0] = unpack_pair(ldsw(st, va[mb][0]), vsh[mb][0], vm[mb][0]);
            vf[mb][1] = unpack_pair(ldsw(st, va[mb][1]), vsh[mb][1], vm[mb][1]);
            vf[mb][2] = unpack_pair(ldsw(st, va[mb][0] + vstep), vsh[mb][0], vm[mb][0]);
            vf[mb][3] = unpack_pair(ldsw(st, va[mb][1] + vstep), vsh[mb][1], vm[mb][1]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the value warp is done with the stage
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&pF[pw]), (uint32_t)(hand & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
      uint32_t bp[NB][2];
      float corr[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        ldsm_x2_t(pa + nb * 16, bp[nb][0], bp[nb][1]);
        corr[nb] = pcorr[nb * 4 + tig];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&pE[pw]));
      ++hand;
      // accumulator columns 2tig, 2tig+1 are head tig (+4 nb). Each tile's products are summed by the MMA from
      // zero and folded into the running sums by round-to-nearest FMAs (acc = acc * corr + tile): accumulating
      // inside the MMA across tiles biases the sums of these positive terms by about 2^-23 per tile, which the
      // near-cancellation of Z and A in the output can magnify a hundredfold.
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        if (mb < nmb) {
          uint32_t af[4];
          if constexpr (NB == 1) {
            af[0] = vf[mb][0], af[1] = vf[mb][1], af[2] = vf[mb][2], af[3] = vf[mb][3];
          } else {
            af[0] = unpack_pair(ldsw(st, va[mb][0]), vsh[mb][0], vm[mb][0]);
            af[1] = unpack_pair(ldsw(st, va[mb][1]), vsh[mb][1], vm[mb][1]);
            af[2] = unpack_pair(ldsw(st, va[mb][0] + vstep), vsh[mb][0], vm[mb][0]);
            af[3] = unpack_pair(ldsw(st, va[mb][1] + vstep), vsh[mb][1], vm[mb][1]);
          }
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            float tile[4];
            mma_f16_zero(tile, af, bp[nb][0], bp[nb][1]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc_o[mb][nb][e] = fmaf(acc_o[mb][nb][e], corr[nb], tile[e]);
          }
        }
      }
      if constexpr (NB != 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // the value warp is done with the stage
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int h = tig + 4 * nb;
      if (h < g) {
        float* w = ws + (pw * 8 + h) * PSTR;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          if (mb < nmb) {
            w[4 + mb * 16 + gid] = acc_o[mb][nb][0] + acc_o[mb][nb][1];
            w[4 + mb * 16 + gid + 8] = acc_o[mb][nb][2] + acc_o[mb][nb][3];
          }
        }
      }
    }
  }

  __syncthreads();
  if (s_abort) {  // drain the copies this CTA may still have in flight, then leave
    if (tid == 0) {
      const int issued = s_issued;
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % NS]), (uint32_t)((i / NS) & 1), a.wait_ns);
    }
    __syncthreads();
    return;
  }

  // ================= epilogue: this split's partial, mapped to the original basis =================
  // N_h[k] = Z_h w_k + sum_j T'[j][k] A_h[j] with T'[j][k] = T_V[j][k] sigma_j 2^-b_j and w_k = sum_{b_j>0} T_V[j][k]
  // sigma_j, so that o_h[k] = base_k + (sum over splits e_s N_s,h[k]) / (sum over splits e_s L_s,h).
  float* Tsc = reinterpret_cast<float*>(smem);                           // [nzV][128]
  float* mA = reinterpret_cast<float*>(smem + L.epi_merged);             // [8][128]
  float* mS = mA + MAX_G * D;                                            // M[8], L[8], Z[8]
  if (tid == 0 && nzV > 0) {
    fence_proxy_async_smem();
    mbar_expect_tx(smem_u32(tbar), (uint32_t)nzV * D * 4);
    bulk_g2s(smem_u32(Tsc), TV.Tsc + (size_t)set * D * D, (uint32_t)nzV * D * 4, smem_u32(tbar));
  }
  __syncthreads();
  {
    const int acols = 4 + nmb * 16;
    for (int idx = tid; idx < g * acols; idx += DTHREADS) {
      const int h = idx / acols, cidx = idx - h * acols;
      if (cidx == 3) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < DWARPS; ++w) M = fmaxf(M, ws[(w * 8 + h) * PSTR]);
      if (cidx == 0) {
        mS[h] = M;
        continue;
      }
      float val = 0.f;
#pragma unroll
      for (int w = 0; w < DWARPS; ++w) {
        const float mw = ws[(w * 8 + h) * PSTR];
        const float e = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        val = fmaf(e, ws[(w * 8 + h) * PSTR + cidx], val);
      }
      if (cidx == 1) mS[MAX_G + h] = val;
      else if (cidx == 2) mS[2 * MAX_G + h] = val;
      else mA[h * D + cidx - 4] = val;
    }
  }
  bool okw = true;
  if (nzV > 0) okw = mbar_wait_bounded(smem_u32(tbar), 0u, a.wait_ns);
  if (!okw && tid == 0) mbar_wait_bounded(smem_u32(tbar), 0u, a.wait_ns);  // drain before leaving
  if (__syncthreads_or(!okw)) return;
  float* part = a.part + ((size_t)bh * a.splits + split) * g * PSTR;
  static_assert(DTHREADS / 32 >= MAX_G && 4 * 32 == D, "a warp per query head, four original channels a lane");
  if (warp < g) {  // warp h: N_h[k] for k = 4 lane .. 4 lane + 3, one 128-bit row segment of T' per rotated channel
    const int h = warp;
    const float4 w4 = reinterpret_cast<const float4*>(TV.wsum + (size_t)set * D)[lane];
    const float zh = mS[2 * MAX_G + h];
    float4 n = make_float4(zh * w4.x, zh * w4.y, zh * w4.z, zh * w4.w);
    const float* ah = mA + h * D;
#pragma unroll 4
    for (int jj = 0; jj < nzV; ++jj) {
      const float4 t = reinterpret_cast<const float4*>(Tsc + jj * D)[lane];
      const float aj = ah[jj];
      n.x = fmaf(t.x, aj, n.x);
      n.y = fmaf(t.y, aj, n.y);
      n.z = fmaf(t.z, aj, n.z);
      n.w = fmaf(t.w, aj, n.w);
    }
    reinterpret_cast<float4*>(part + h * PSTR + 4)[lane] = n;
  }
  if (tid < g) {
    part[tid * PSTR + 0] = mS[tid];
    part[tid * PSTR + 1] = mS[MAX_G + tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.cnt[bh], 1u) == (unsigned)(a.splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ======== last CTA of (b, kh): weighted sum of the split partials ========
  // The partials arrive in shared memory by bulk copies (chunks of splits); warp h (< g) keeps head h's running
  // maximum M_h and L_h = sum e_s l_s with the weights e_s = 2^(m_s - M_h) (lanes over the chunk's splits,
  // shuffle reductions); every thread then adds its outputs' sum e_s N_s from shared memory.
  float* esc = reinterpret_cast<float*>(smem + L.tail_reserve);  // [MAX_SPLITS][8] weights of the chunk
  float* hst = esc + MAX_SPLITS * MAX_G;                         // L[8], rescale of the running sums[8]
  const float* pb = a.part + (size_t)bh * a.splits * g * PSTR;
  const int S = a.splits;
  const uint32_t per_split = (uint32_t)g * PSTR * 4;
  const int chunk_splits = max(1, min(S, min((int)(L.tail_reserve / per_split), MAX_SPLITS)));
  constexpr int ITEMS_PER_THREAD = MAX_G * D / DTHREADS;
  constexpr int SPL = MAX_SPLITS / 32;  // splits per lane within a chunk
  float accN[ITEMS_PER_THREAD];
#pragma unroll
  for (int r = 0; r < ITEMS_PER_THREAD; ++r) accN[r] = 0.f;
  float M_run = -INFINITY, L_run = 0.f;  // warp h's running state of head h
  uint32_t tphase = nzV > 0 ? 1u : 0u;   // phase 0 of tbar went to the T' copy when there was one
  fence_proxy_async_global();
  const float* cp = reinterpret_cast<const float*>(smem);
  for (int c0s = 0; c0s < S; c0s += chunk_splits) {
    const int n = min(chunk_splits, S - c0s);
    __syncthreads();  // previous chunk consumed
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_expect_tx(smem_u32(tbar), (uint32_t)n * per_split);
      bulk_g2s(smem_u32(smem), pb + (size_t)c0s * g * PSTR, (uint32_t)n * per_split, smem_u32(tbar));
    }
    const bool okc = mbar_wait_bounded(smem_u32(tbar), tphase, a.wait_ns);
    if (!okc && tid == 0) mbar_wait_bounded(smem_u32(tbar), tphase, a.wait_ns);  // drain before leaving
    tphase ^= 1u;
    if (!__syncthreads_and(okc)) return;
    if (warp < g) {
      const int h = warp;
      float ms[SPL];
      float cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const int sp = lane + 32 * i;
        ms[i] = sp < n ? cp[(sp * g + h) * PSTR] : -INFINITY;
        cm = fmaxf(cm, ms[i]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float Mn = fmaxf(M_run, cm);
      const float sc = (M_run == Mn) ? 1.f : exp2f(M_run - Mn);
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const int sp = lane + 32 * i;
        if (sp < n) {
          const float e = ms[i] == -INFINITY ? 0.f : exp2f(ms[i] - Mn);
          esc[sp * MAX_G + h] = e;
          l = fmaf(e, cp[(sp * g + h) * PSTR + 1], l);
        }
      }
      L_run = fmaf(L_run, sc, warp_sum(l));
      M_run = Mn;
      if (lane == 0) {
        hst[h] = L_run;
        hst[MAX_G + h] = sc;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ITEMS_PER_THREAD; ++r) {
      const int it = tid + r * DTHREADS;
      if (it < g * D) {
        const int h = it >> 7, k = it & (D - 1);
        float acc = accN[r] * hst[MAX_G + h];
        for (int sp = 0; sp < n; ++sp) acc = fmaf(esc[sp * MAX_G + h], cp[(sp * g + h) * PSTR + 4 + k], acc);
        accN[r] = acc;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < ITEMS_PER_THREAD; ++r) {
    const int it = tid + r * DTHREADS;
    if (it < g * D) {
      const int h = it >> 7, k = it & (D - 1);
      const float Lh = hst[h];
      a.out[((size_t)b * a.Hq + (size_t)kh * g + h) * D + k] =
          Lh > 0.f ? TV.base[(size_t)set * D + k] + accN[r] / Lh : 0.f;
    }
  }
  if (tid == 0) a.cnt[bh] = 0u;
}

static void split_plan(int B, int Hkv, int64_t T_cap, int device, int tile, int per_sm, int max_splits,
                       int* splits, int* chunk) {
  const long long bh = (long long)B * Hkv;
  const long long tiles = (T_cap + tile - 1) / tile;
  long long sp = ((long long)per_sm * sm_count(device) + bh - 1) / bh;
  sp = std::max(1LL, std::min(std::min(sp, tiles), (long long)max_splits));
  const long long ct = (tiles + sp - 1) / sp;
  *splits = (int)((tiles + ct - 1) / ct);
  *chunk = (int)(ct * tile);
}

DecodeLayout decode_layout(int B, int Hkv, int Hq, int64_t T_cap, int device) {
  DecodeLayout L{};
  split_plan(B, Hkv, T_cap, device, DT, 2, MAX_SPLITS, &L.splits, &L.chunk);
  const size_t bh = (size_t)B * Hkv;
  const int g = Hq / Hkv;
  size_t o = 0;
  L.off_qa = o;
  o = align256(o + bh * 16 * D * sizeof(__half));
  L.off_qc = o;
  o = align256(o + bh * QP_PARTS * QPC * sizeof(float));
  L.off_cnt = o;
  o = align256(o + bh * sizeof(unsigned));
  L.off_part = o;
  o = align256(o + bh * (size_t)L.splits * g * PSTR * sizeof(float));
  L.total = o;
  return L;
}

// record lengths with a compile-time decode kernel (equal key and value budgets of 1.25 - 4 bits/element)
static int compile_time_record_words(int RK, int RV) {
  if (RK != RV) return 0;
  switch (RK) {
    case 5: case 8: case 11: case 12: case 16: return RK;
    default: return 0;
  }
}

template <int NB, int RT, bool PIPE>
static cudaError_t launch_decode_kernel(cudaLaunchConfig_t& cfg, const ParamsDev& P, const DecArgs& a) {
  const cudaError_t e = ensure_dyn_smem((const void*)decode_kernel<NB, RT, PIPE>, cfg.dynamicSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<NB, RT, PIPE>, P, a);
}

template <int NB, bool PIPE>
static cudaError_t launch_decode_nb(cudaLaunchConfig_t& cfg, const ParamsDev& P, const DecArgs& a, int rt) {
  switch (rt) {
    case 5: return launch_decode_kernel<NB, 5, PIPE>(cfg, P, a);
    case 8: return launch_decode_kernel<NB, 8, PIPE>(cfg, P, a);
    case 11: return launch_decode_kernel<NB, 11, PIPE>(cfg, P, a);
    case 12: return launch_decode_kernel<NB, 12, PIPE>(cfg, P, a);
    case 16: return launch_decode_kernel<NB, 16, PIPE>(cfg, P, a);
    default: return launch_decode_kernel<NB, 0, PIPE>(cfg, P, a);
  }
}

kv_status launch_decode(const ParamsDev& P, const kv_cache& c, const void* q, int B, int Hq,
                        const int32_t* seq_lens, float scale, float* out, void* ws, const DecodeLayout& L,
                        cudaStream_t s) {
  DecArgs a;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.rec[0] = c.k_rec;
  a.rec[1] = c.v_rec;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_lens = seq_lens;
  a.qa = reinterpret_cast<__half*>(w + L.off_qa);
  a.qc = reinterpret_cast<float*>(w + L.off_qc);
  a.cnt = reinterpret_cast<unsigned*>(w + L.off_cnt);
  a.part = reinterpret_cast<float*>(w + L.off_part);
  a.out = out;
  a.T_cap = c.T_cap;
  a.wait_ns = g_wait_limit_ns;
  a.B = B;
  a.Hkv = c.Hkv;
  a.Hq = Hq;
  a.g = Hq / c.Hkv;
  a.per_seq = c.per_seq_params;
  a.splits = L.splits;
  a.chunk = L.chunk;
  const int rt = compile_time_record_words(P.t[0].r_words, P.t[1].r_words);
  a.stages = ring_stages_for(P.t[0].r_words, P.t[1].r_words);
  a.scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t qc = {};
    qc.gridDim = dim3(c.Hkv, B, QP_PARTS);
    qc.blockDim = dim3(QP_THREADS);
    qc.dynamicSmemBytes = 0;
    qc.stream = s;
    qc.attrs = pdl;
    qc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&qc, qprep_kernel, P, a);
    if (e != cudaSuccess) {
      set_error("qprep_kernel launch: %s", cudaGetErrorString(e));
      return KV_ERR_CUDA;
    }
  }
  kv_status st = launch_check("qprep_kernel");
  if (st != KV_OK) return st;
  const int nb = a.g <= 4 ? 1 : 2;
  const size_t smem = decode_smem(P.t[0].r_words, P.t[1].r_words, a.stages, nb).total;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.splits, c.Hkv, B);
  cfg.blockDim = dim3(DTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  // the pipelined key loop processes all eight key channel blocks: taken when every set needs at least seven
  const bool pipe = nb == 1 && P.t[0].min_nz > 6 * 16;
  const cudaError_t e = nb == 1 ? (pipe ? launch_decode_nb<1, true>(cfg, P, a, rt) : launch_decode_nb<1, false>(cfg, P, a, rt))
                                : launch_decode_nb<2, false>(cfg, P, a, rt);
  if (e != cudaSuccess) {
    set_error("decode_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return launch_check("decode_kernel");
}

}  // namespace kvtc
