// Decode over packed records: the split-K flash-decode kernel (with the q preparation in its prologue) and its
// launcher. Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
//
// Method: "SPHERICAL KV ..." page, third abstract (NOVA-KV): decode re-reads the whole cache at every step and is
// bandwidth-bound, so the cost of turning a stored code back into something attention can use has to stay small.
// Here no dequantised key or value is ever formed: the codes enter fp16 tensor-core MMAs directly and every
// per-channel affine term of the dequantisation is folded into per-head constants.
//
// Code extraction. A slot (key: channels 2k, 2k+1 of one token; value: channel j of the two tokens of a record)
// holds its two codes at bits [r, r + b) of the low and the high half of one code word. Rotating the word left by
// (10 - w - r) mod 32 (w: the slot's width, b <= w) puts them at bits [10 - w, 10 - w + b) and [26 - w, ...);
// masking them and OR-ing in the fp16 exponent of 1.0 gives the fp16 pair (1 + c_lo 2^-w, 1 + c_hi 2^-w), exact
// for w <= 10: two instructions per MMA operand register after the shared-memory load.
//
// Logits (base 2), per head h, token t, with Q_j = a log2(e) (T_K q_h)_j sigma_j and w_j the slot width of channel
// j (b_j its code width; w_j = b_j except for a narrower channel sharing a key slot):
//   l_t = C0 + z_t C1 + s_t (sum_j Q_j 2^(w_j - b_j) A_tj - C2),  A_tj = 1 + c_tj 2^-w_j,
//   C0 = a log2(e) q.(T_K^T mu),  C1 = sum_{b_j>0} Q_j = a log2(e) q.w,  C2 = sum_{b_j>0} Q_j (2^(w_j - b_j) -
//   2^(-b_j - 1)) = a log2(e) q.w2  (w, w2: the key table's folded vectors),
// which is a log2(e) q.k^ for k^ = T_K^T y^, y^_j = mu_j + sigma_j (z + (c_j + 1/2) s 2^-b_j).
// Values, per head, with weights p_t (unnormalised softmax) and W_t = p_t s_t (value slots have w_j = b_j):
//   sum_t p_t y^_tj = l mu_j + sigma_j (Z - (1 - 2^(-b_j - 1)) S + M_j),  M_j = sum_t W_t A_tj,
//   Z = sum_t p_t z_t, S = sum_t W_t, l = sum_t p_t,
// so the original-basis output is o_k = (T_V^T mu)_k + (Z w_k - S w2_k + sum_j T'_jk M_j) / l with
// T'_jk = T_V[j][k] sigma_j, w_k = sum_j T'_jk, w2_k = sum_j T'_jk (1 - 2^(-b_j - 1)) (sums over b_j > 0).
// Each split leaves (m, l, Z, S, M) in the rotated basis; the last split to finish merges them with their softmax
// weights and maps the result to the original basis once.
#pragma once
#include <type_traits>

namespace kvtc {

// ======================================================================================================
// decode over packed records
// ======================================================================================================
constexpr int PSTR = 132;              // floats per (split, head) partial: m, l, Z, S, M[128]
constexpr int WT = 32;                 // tokens of a warp pair per ring stage
constexpr int RING_BUDGET = 128 * 1024;
constexpr int MAX_STAGES = 8;
constexpr int MAX_SPLITS = 256;
constexpr int TAIL_RESERVE = MAX_SPLITS * MAX_G * 4 + 4 * MAX_G * 4;  // split weights, head state
constexpr int HC = 4;                  // per-head constants: C0, C1, C2, 2^-e

// warp pairs (a key warp and a value warp) per CTA: eight with one 8-column block (128 registers a thread, one
// 16-warp CTA per SM), four with two (the heads' operands and sums need more registers)
__host__ __device__ constexpr int dec_pairs(int nb) { return nb == 1 ? 8 : 4; }
__host__ __device__ constexpr int dec_threads(int nb) { return 64 * dec_pairs(nb); }
__host__ __device__ constexpr int dec_stage_tokens(int nb) { return WT * dec_pairs(nb); }
static_assert(dec_threads(2) / 32 >= MAX_G, "one warp per query head of a group in the merge");

struct DecArgs {
  const uint32_t* rec[2];
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  unsigned* cnt;    // [B*Hkv] arrival counters: zero before a call, left at zero after it
  float* part;      // [B*Hkv][splits][g][PSTR] split partials
  float* out;       // [B][Hq][128]
  long long T_cap;
  long long wait_ns;
  int B, Hkv, Hq, g, per_seq, splits, stages;
  float scale_log2;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__host__ __device__ __forceinline__ uint32_t align128u(uint32_t x) { return (x + 127u) & ~127u; }

// P hand-off buffer of one warp pair and one slot: the softmax weights p (fp32) [2 m-tiles][4 NB heads][24] (16
// tokens, rows padded to 24 floats so that both the key warp's stores and the value warp's 64-bit loads are free
// of bank conflicts), then the NB x 4 rescale factors.
constexpr int PROW = 24;
__host__ __device__ constexpr uint32_t pbuf_bytes(int nb) { return 2u * 4u * nb * PROW * 4u + 16u * nb; }

struct DecSmem {  // byte offsets into the dynamic shared memory of decode_kernel
  uint32_t stage_bytes, qa, hc, pbuf, epi, chunks, tail_reserve, total;
};

// main loop: ring | q' operands [16][128] fp16 | per-head constants | P buffers (pairs x 2 slots)
// prologue scratch from epi: q [8][128] f32, partial q~ [parts][8][128] f32, coefficient scales [8]
// epilogue: per-warp-pair partials from epi
// tail (last CTA): T'_V rows [0, 64 KB) | split partial chunks [64 KB, tail_reserve) | merged partial and the
//   per-split weights and per-head state in the reserve at the end
__host__ __device__ inline DecSmem decode_smem(int RK, int RV, int stages, int nb) {
  DecSmem s;
  const int pairs = dec_pairs(nb), parts = dec_threads(nb) / D;
  s.stage_bytes = (uint32_t)dec_stage_tokens(nb) * (RK + RV) * 4u;
  s.qa = align128u(stages * s.stage_bytes);
  s.hc = s.qa + 16u * D * 2u;
  s.pbuf = align128u(s.hc + MAX_G * HC * 4u);
  const uint32_t main_end = s.pbuf + pairs * 2u * pbuf_bytes(nb);
  s.epi = align128u(main_end);
  const uint32_t prologue_end = s.epi + (MAX_G * D + parts * MAX_G * D + MAX_G) * 4u;
  const uint32_t epi_end = s.epi + pairs * 8u * PSTR * 4u;
  s.chunks = (uint32_t)D * D * 4u;
  uint32_t end = prologue_end > epi_end ? prologue_end : epi_end;
  const uint32_t tail_min = s.chunks + 8u * MAX_G * PSTR * 4u;  // room for eight splits' partials at least
  end = end > tail_min ? end : tail_min;
  s.tail_reserve = align128u(end);
  s.total = s.tail_reserve + (MAX_G * PSTR + 4 * MAX_G) * 4u + TAIL_RESERVE;
  return s;
}

__host__ __device__ constexpr int ring_stages_for(int RK, int RV, int nb) {
  return (RING_BUDGET / (dec_stage_tokens(nb) * (RK + RV) * 4)) > MAX_STAGES ? MAX_STAGES
         : (RING_BUDGET / (dec_stage_tokens(nb) * (RK + RV) * 4)) < 2      ? 2
                                                                          : RING_BUDGET / (dec_stage_tokens(nb) * (RK + RV) * 4);
}

// Four shared-memory words at a 32-bit shared address and three further multiples of a byte stride (an immediate
// when STRIDE > 0). Volatile, so that they stay after the barrier wait that makes the stage's bytes visible.
template <int STRIDE>
__device__ __forceinline__ void lds_x4(uint32_t addr, uint32_t stride, uint32_t& v0, uint32_t& v1, uint32_t& v2,
                                       uint32_t& v3) {
  if constexpr (STRIDE > 0) {
    asm volatile(
        "ld.shared.b32 %0, [%4];\n\tld.shared.b32 %1, [%4+%5];\n\tld.shared.b32 %2, [%4+%6];\n\t"
        "ld.shared.b32 %3, [%4+%7];"
        : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
        : "r"(addr), "n"(STRIDE), "n"(2 * STRIDE), "n"(3 * STRIDE));
  } else {
    asm volatile(
        "ld.shared.b32 %0, [%4];\n\tld.shared.b32 %1, [%5];\n\tld.shared.b32 %2, [%6];\n\t"
        "ld.shared.b32 %3, [%7];"
        : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
        : "r"(addr), "r"(addr + stride), "r"(addr + 2 * stride), "r"(addr + 3 * stride));
  }
}

// One slot as an fp16 pair (1 + c_lo 2^-w, 1 + c_hi 2^-w): rotate the code word left by rot (the low five bits of
// desc), keep the two code fields, put the exponent of 1.0 under them.
__device__ __forceinline__ uint32_t slot_f16x2(uint32_t word, uint32_t desc, uint32_t mask) {
  return (__funnelshift_l(word, word, desc) & mask) | 0x3C003C00u;
}

// Slot descriptor for the decode: byte offset of the code word within a ring stage (bits 5..) and the rotation
// (bits 0..4); mask of the two code fields after the rotation. w: slot width; b_lo, b_hi: code widths.
__device__ __forceinline__ void slot_decode_desc(uint32_t stage_off, uint32_t r, uint32_t w, uint32_t b_lo,
                                                 uint32_t b_hi, uint32_t& desc, uint32_t& mask) {
  desc = (stage_off << 5) | ((10u - w - r) & 31u);
  mask = w ? ((((1u << b_lo) - 1u) << (10u - w)) | (((1u << b_hi) - 1u) << (26u - w))) : 0u;
}

// RK_, RV_ > 0: compile-time record lengths (ring stage size and count, token row offsets as immediates).
// NB: 8-column blocks of the MMA's n dimension (4 heads each, fp16 hi and lo columns). NBLK: 16-channel blocks
// processed per tensor (blocks past a set's last nonzero-width channel hold zero masks and zero coefficients).
template <int NB, int RK_, int RV_, int NBLK>
__global__ void __launch_bounds__(dec_threads(NB), 1) decode_kernel(ParamsDev P, DecArgs a) {
  constexpr int DW = dec_pairs(NB), DTHREADS = dec_threads(NB), DT = dec_stage_tokens(NB);
  constexpr int QPARTS = DTHREADS / D, KQ = D / QPARTS;  // q preparation: threads per channel, k's per thread
  extern __shared__ __align__(128) uint8_t smem[];
  // barriers live outside the dynamic region, which the epilogue and the tail reuse wholesale
  __shared__ __align__(8) uint64_t full[MAX_STAGES], pF[DW][2], pE[DW][2], tbar_s, vbar_s;
  __shared__ unsigned rel[MAX_STAGES];  // warps done with the stage in each ring slot
  __shared__ int s_abort, s_last, s_issued;
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int bh = b * a.Hkv + kh;
  const int set = a.per_seq ? bh : kh;
  const TensorDev& TK = P.t[0];
  const TensorDev& TV = P.t[1];
  const int RK = RK_ ? RK_ : TK.r_words, RV = RV_ ? RV_ : TV.r_words;
  constexpr int NS_CT = RK_ ? ring_stages_for(RK_, RV_, NB) : 0;
  const int NS = RK_ ? NS_CT : a.stages, g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const size_t so = (size_t)set * D;
  const int nzK = TK.nz[set], nzV = TV.nz[set];
  const int nkb = (nzK + 15) >> 4, nmb = (nzV + 15) >> 4;
  const DecSmem L = decode_smem(RK, RV, NS, NB);
  const uint32_t stage_bytes = (uint32_t)DT * (RK + RV) * 4u;
  uint64_t* tbar = &tbar_s;
  __half* qa = reinterpret_cast<__half*>(smem + L.qa);  // [16 columns][128 channels]
  float* hc = reinterpret_cast<float*>(smem + L.hc);    // [8 heads][HC]

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      rel[s] = 0u;
    }
    for (int p = 0; p < DW; ++p)
      for (int sl = 0; sl < 2; ++sl) {
        mbar_init(smem_u32(&pF[p][sl]), 1);
        mbar_init(smem_u32(&pE[p][sl]), 1);
      }
    mbar_init(smem_u32(tbar), 1);
    mbar_init(smem_u32(&vbar_s), 1);
    fence_mbar_init();
    s_abort = 0;
    s_issued = 0;
  }
  // ---- parameters only (nothing a previous kernel writes), all in one round of loads ----
  uint32_t sd[NBLK][2], sm[NBLK][2];  // slot descriptors of this warp's role
  if (warp < DW) {  // key warp: pair 8 kb + 4 i + tig of token rows WT pw + gid (+ 8, 16, 24)
#pragma unroll
    for (int kb = 0; kb < NBLK; ++kb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t dk = kb < nkb ? __ldg(TK.slots + so + 8 * kb + 4 * i + tig) : 0u;
        const uint32_t b0 = (dk >> 16) & 255u, b1 = dk >> 24, w = b0 > b1 ? b0 : b1;
        const uint32_t off = (uint32_t)(WT * warp + gid) * RK * 4u + 4u * (1u + (dk & 255u));
        slot_decode_desc(off, (dk >> 8) & 255u, w, b0, b1, sd[kb][i], sm[kb][i]);
      }
  } else {          // value warp: channel 16 mb + 8 i + gid of token-pair records (WT/2) pw + tig (+ 4, 8, 12)
#pragma unroll
    for (int mb = 0; mb < NBLK; ++mb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t dv = mb < nmb ? __ldg(TV.slots + so + 16 * mb + 8 * i + gid) : 0u;
        const uint32_t bw = (dv >> 16) & 255u;
        const uint32_t off = (uint32_t)DT * RK * 4u + (uint32_t)((WT / 2) * (warp - DW) + tig) * 2u * RV * 4u +
                             4u * (2u + (dv & 255u));
        slot_decode_desc(off, (dv >> 8) & 255u, bw, bw, bw, sd[mb][i], sm[mb][i]);
      }
  }
  // q preparation: this thread's slice of T^T (rows KQ part .. KQ part + KQ - 1, column j), channel j's sigma and
  // widths; warp h < 8: the folded key vectors at its lane's four entries
  const int qj = tid & (D - 1), qpart = tid / D;
  float tt[KQ];
  {
    const float* TTc = TK.TT + so * D + (size_t)(KQ * qpart) * D + qj;
#pragma unroll
    for (int kk = 0; kk < KQ; ++kk) tt[kk] = __ldg(TTc + (size_t)kk * D);
  }
  const float q_sg = __ldg(TK.sigma + so + qj);
  const int q_bj = __ldg(TK.widths + so + qj), q_bp = __ldg(TK.widths + so + (qj ^ 1));
  float4 kb4 = make_float4(0.f, 0.f, 0.f, 0.f), kw4 = kb4, kv4 = kb4;
  float ksmax = 0.f;
  if (warp < MAX_G) {
    kb4 = reinterpret_cast<const float4*>(TK.base + so)[lane];
    kw4 = reinterpret_cast<const float4*>(TK.wsum + so)[lane];
    kv4 = reinterpret_cast<const float4*>(TK.wsum2 + so)[lane];
    ksmax = __ldg(TK.smax + set);
  }
  __syncthreads();

  // The previous kernel of the stream (an append, say) may still be running: q and the records are read only
  // after it has completed.
  pdl_wait();

  // this sequence's tokens spread over all the splits: chunks of whole stages sized from its own length, so a
  // short sequence in a long cache (or in a ragged batch) keeps every split busy
  const long long Lseq = max(0LL, min((long long)a.seq_lens[b], a.T_cap));
  const long long chunk = ((Lseq + a.splits - 1) / a.splits + DT - 1) / DT * DT;
  const long long t0 = min((long long)split * chunk, Lseq);
  const long long t1 = min(t0 + chunk, Lseq);
  const int ntiles = (int)((t1 - t0 + DT - 1) / DT);
  const int n_in = (int)(t1 - t0);

  // ---- record stages stream into the ring by bulk copies: thread 0 fills the ring, then the last of the 2 DW warps
  // to release a slot refills it at once with the stage NS further on ----
  const uint32_t* krec = a.rec[0] + (size_t)bh * a.T_cap * RK;
  const uint32_t* vrec = a.rec[1] + (size_t)bh * a.T_cap * RV;  // two-token records: same bytes per token
  const uint32_t ring = smem_u32(smem);
  auto issue_tile = [&](int i) {
    const int s = i % NS;
    const long long tb = t0 + (long long)i * DT;
    long long n = min((long long)DT, t1 - tb);
    n = min((n + 3) & ~3LL, a.T_cap - tb);
    const uint32_t kbytes = (uint32_t)(n * RK * 4), vbytes = (uint32_t)(n * RV * 4);
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t dst = ring + (uint32_t)s * stage_bytes;
    mbar_expect_tx(bar, kbytes + vbytes);
    bulk_g2s(dst, krec + tb * RK, kbytes, bar);
    bulk_g2s(dst + DT * RK * 4, vrec + tb * RV, vbytes, bar);
  };
  // this warp is done reading stage i: the last warp to say so issues stage i + NS into the same slot (its
  // acquire-release count orders every warp's reads of the slot before the refill's writes)
  auto release_stage = [&](int i) {
    __syncwarp();
    if (lane == 0) {
      const int s = i % NS;
      unsigned old;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(&rel[s])) : "memory");
      if (old == 2u * DW - 1u) {
        rel[s] = 0u;
        if (i + NS < ntiles) {
          fence_proxy_async_smem();
          issue_tile(i + NS);
          atomicMax(&s_issued, i + NS + 1);
        }
      }
    }
  };
  if (tid == 0) {
    if (split == 0 && nzV > 0)  // the merge of this (sequence, head) reads the scaled T_V rows: warm L2 now
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(TV.Tsc + so * D), "r"((uint32_t)nzV * D * 4)
                   : "memory");
    for (int i = 0; i < NS && i < ntiles; ++i) issue_tile(i);
    s_issued = min(NS, ntiles);
  }

  // ---- q preparation: per-head constants from dot products of q with the folded vectors, then
  // q~ = T_K q and the MMA coefficients Q_j 2^(w_j - b_j) 2^e_h as fp16 hi + lo pairs ----
  {
    float* qs = reinterpret_cast<float*>(smem + L.epi);  // [8][128]
    float* red = qs + MAX_G * D;                          // [QPARTS][8][128]
    float* esc = red + QPARTS * MAX_G * D;                // [8] 2^e_h
    if (warp < MAX_G) {  // warp h: head h's row of q, its norm and its three dot products
      const int h = warp;
      float4 qv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (h < g) {
        const uint2 u = reinterpret_cast<const uint2*>(a.q + ((size_t)b * a.Hq + (size_t)kh * g + h) * D)[lane];
        qv = make_float4(bf16_bits_f(u.x & 0xFFFFu), bf16_bits_f(u.x >> 16), bf16_bits_f(u.y & 0xFFFFu),
                         bf16_bits_f(u.y >> 16));
      }
      reinterpret_cast<float4*>(qs + h * D)[lane] = qv;
      const float n2 = warp_sum(qv.x * qv.x + qv.y * qv.y + qv.z * qv.z + qv.w * qv.w);
      const float c0 = warp_sum(qv.x * kb4.x + qv.y * kb4.y + qv.z * kb4.z + qv.w * kb4.w);
      const float c1 = warp_sum(qv.x * kw4.x + qv.y * kw4.y + qv.z * kw4.z + qv.w * kw4.w);
      const float c2 = warp_sum(qv.x * kv4.x + qv.y * kv4.y + qv.z * kv4.z + qv.w * kv4.w);
      if (lane == 0) {
        // 2^e_h scales the coefficients so that the largest (<= |a log2 e| |q_h| smax) sits near 2^12..2^14: the
        // fp16 hi + lo pair then keeps about 22 bits for every channel that matters; the logit sum is multiplied
        // by 2^-e_h
        const float bound = fabsf(a.scale_log2) * sqrtf(n2) * ksmax;
        int e = 0;
        if (bound > 0.f && bound <= 3.0e38f) {
          int ex;
          frexpf(bound, &ex);  // bound < 2^ex
          e = min(max(14 - ex, -120), 120);
        }
        hc[h * HC + 0] = a.scale_log2 * c0;
        hc[h * HC + 1] = a.scale_log2 * c1;
        hc[h * HC + 2] = a.scale_log2 * c2;
        hc[h * HC + 3] = exp2i(-e);
        esc[h] = exp2i(e);
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < MAX_G; ++h) {  // q~_h[j] over k in [KQ part, KQ part + KQ)
      float acc = 0.f;
      if (h < g) {
        const float4* q4 = reinterpret_cast<const float4*>(qs + h * D + KQ * qpart);
#pragma unroll
        for (int k4 = 0; k4 < KQ / 4; ++k4) {
          const float4 v = q4[k4];
          acc = fmaf(tt[4 * k4], v.x, acc);
          acc = fmaf(tt[4 * k4 + 1], v.y, acc);
          acc = fmaf(tt[4 * k4 + 2], v.z, acc);
          acc = fmaf(tt[4 * k4 + 3], v.w, acc);
        }
      }
      red[(qpart * MAX_G + h) * D + qj] = acc;
    }
    __syncthreads();
    if (tid < D) {
      const int j = qj, bj = q_bj, wj = q_bj > q_bp ? q_bj : q_bp;  // slot width of the channel pair
      const float f = bj > 0 ? a.scale_log2 * q_sg * exp2i(wj - bj) : 0.f;
#pragma unroll
      for (int h = 0; h < MAX_G; ++h) {
        float qt = 0.f;
#pragma unroll
        for (int p = 0; p < QPARTS; ++p) qt += red[(p * MAX_G + h) * D + j];
        const float c = h < g ? qt * f * esc[h] : 0.f;
        const __half hi = __float2half_rn(c);
        const __half lo = __float2half_rn(c - __half2float(hi));
        qa[(2 * h) * D + j] = hi;
        qa[(2 * h + 1) * D + j] = lo;
      }
    }
    __syncthreads();
  }

  // ============ warp pairs: key warp pw and value warp pw + DW own tokens [32 pw, 32 pw + 32) of every stage ============
  const int pw = warp % DW;
  uint8_t* const pbase = smem + L.pbuf + (size_t)pw * 2 * pbuf_bytes(NB);
  float* ws = reinterpret_cast<float*>(smem + L.epi);  // [DW][8][PSTR] (the prologue scratch is dead)
  constexpr uint32_t PCORR = 2u * 4u * NB * PROW * 4u;  // byte offset of the rescale factors in a P buffer
  if (warp < DW) {
    // ---------------- key warp: logits (MMA over the key codes), online softmax, p to the value warp ----------------
    uint32_t qb[NBLK][NB][2];  // B operand: coefficients, k = channels 16 kb + 2 tig (+1, +8, +9), n = column gid
    {
      const uint32_t* qa32 = reinterpret_cast<const uint32_t*>(qa);
#pragma unroll
      for (int kb = 0; kb < NBLK; ++kb)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int col = nb * 8 + gid;
          qb[kb][nb][0] = qa32[(col * D + kb * 16 + 2 * tig) >> 1];
          qb[kb][nb][1] = qa32[(col * D + kb * 16 + 8 + 2 * tig) >> 1];
        }
    }
    float C0[NB], C1[NB], C2[NB], qsc[NB], m_run[NB], l_run[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int h = tig + 4 * nb;
      C0[nb] = hc[h * HC + 0];
      C1[nb] = hc[h * HC + 1];
      C2[nb] = hc[h * HC + 2];
      qsc[nb] = hc[h * HC + 3];
      m_run[nb] = -INFINITY;
      l_run[nb] = 0.f;
    }
    const uint32_t kzo = (uint32_t)(WT * pw + gid) * RK * 4u;
    constexpr int KSTR = RK_ ? 8 * RK_ * 4 : 0;  // token rows +8
    const uint32_t kstr = 8u * RK * 4u;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NS;
      const uint32_t sb = ring + (uint32_t)s * stage_bytes;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((i / NS) & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
      // ---- logits: A = key codes (16 tokens x 16 channels) of m-tiles 0 (rows gid, gid + 8) and 1 (+16); two
      // accumulators per m-tile (even and odd channel blocks) halve the MMA dependency chain ----
      float acc[2][2][NB][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            acc[mt][pr][nb][0] = acc[mt][pr][nb][1] = acc[mt][pr][nb][2] = acc[mt][pr][nb][3] = 0.f;
#pragma unroll
      for (int kb = 0; kb < NBLK; ++kb) {
        uint32_t af[2][4];  // rows gid, gid + 8 (m-tile 0), gid + 16, gid + 24 (m-tile 1)
        lds_x4<KSTR>(sb + (sd[kb][0] >> 5), kstr, af[0][0], af[0][1], af[1][0], af[1][1]);
        lds_x4<KSTR>(sb + (sd[kb][1] >> 5), kstr, af[0][2], af[0][3], af[1][2], af[1][3]);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          af[mt][0] = slot_f16x2(af[mt][0], sd[kb][0], sm[kb][0]);
          af[mt][1] = slot_f16x2(af[mt][1], sd[kb][0], sm[kb][0]);
          af[mt][2] = slot_f16x2(af[mt][2], sd[kb][1], sm[kb][1]);
          af[mt][3] = slot_f16x2(af[mt][3], sd[kb][1], sm[kb][1]);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16(acc[mt][kb & 1][nb], af[mt], qb[kb][nb][0], qb[kb][nb][1]);
        }
      }
      // z/s words of this lane's four tokens (rows gid + 8 m) of their key records
      uint32_t kzw[4];
      lds_x4<KSTR>(sb + kzo, kstr, kzw[0], kzw[1], kzw[2], kzw[3]);
      release_stage(i);
      const int r0 = i * DT + WT * pw + gid;  // split-relative token of row m: r0 + 8 m
      float zk[4], sk[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 fk = __half22float2(*reinterpret_cast<const __half2*>(&kzw[m]));
        zk[m] = fk.x;
        sk[m] = fk.y;
      }
      float pv[4][NB];
      float corr[NB];
      // logits, online softmax; FULL: every token of the stage is in the split (no masking)
      auto softmax = [&](auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        bool val[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) val[m] = FULL || r0 + 8 * m < n_in;
        float l[NB][4];
        bool up = false;  // a logit above the running maximum of its head
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float* c0 = acc[m >> 1][0][nb];
            const float* c1 = acc[m >> 1][1][nb];
            const int e = 2 * (m & 1);
            const float r = fmaf((c0[e] + c1[e]) + (c0[e + 1] + c1[e + 1]), qsc[nb], -C2[nb]);
            const float lv = fmaf(sk[m], r, fmaf(zk[m], C1[nb], C0[nb]));
            l[nb][m] = val[m] ? lv : -INFINITY;
            up |= l[nb][m] > m_run[nb];
          }
        if (__any_sync(0xffffffffu, up)) {  // the running maxima move: recompute them across the warp
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            float mt = fmaxf(fmaxf(l[nb][0], l[nb][1]), fmaxf(l[nb][2], l[nb][3]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            const float m_new = fmaxf(m_run[nb], mt);
            corr[nb] = (m_run[nb] == m_new) ? 1.f : ex2_approx(m_run[nb] - m_new);
            m_run[nb] = m_new;
          }
        } else {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) corr[nb] = 1.f;
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float ps = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float e2 = ex2_approx(l[nb][m] - m_run[nb]);
            pv[m][nb] = val[m] ? e2 : 0.f;
            ps += pv[m][nb];
          }
          l_run[nb] = fmaf(l_run[nb], corr[nb], ps);
        }
      };
      if ((i + 1) * DT <= n_in)
        softmax(std::true_type{});
      else
        softmax(std::false_type{});
      // ---- hand p and the rescale factors to the value warp ----
      const int slot = i & 1;
      if (i >= 2 && !__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&pE[pw][slot]),
                                                            (uint32_t)(((i >> 1) - 1) & 1), a.wait_ns, 64))) {
        s_abort = 1;
        break;
      }
      float* pt = reinterpret_cast<float*>(pbase + slot * pbuf_bytes(NB));
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) pt[((m >> 1) * 4 * NB + 4 * nb + tig) * PROW + gid + 8 * (m & 1)] = pv[m][nb];
      if (gid == 0) {
        float* pc = reinterpret_cast<float*>(pbase + slot * pbuf_bytes(NB) + PCORR);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) pc[nb * 4 + tig] = corr[nb];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&pF[pw][slot]));
    }
    // this warp's softmax state into the per-warp partial
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float lsum = l_run[nb];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
      const int h = tig + 4 * nb;
      if (h < g && gid == 0) {
        float* w = ws + (pw * 8 + h) * PSTR;
        w[0] = m_run[nb];
        w[1] = lsum;
      }
    }
  } else {
    // ---------------- value warp: W = p s_V as fp16 hi/lo (the B operand), Z = sum p z_V, S = sum W, and
    // M_j = sum_t W_t A_tj on the MMA (A = value codes) ----------------
    float acc[NBLK][NB][4];
#pragma unroll
    for (int mb = 0; mb < NBLK; ++mb)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mb][nb][e] = 0.f;
    // B fragment of a 16-token m-tile: this lane holds column gid (head gid / 2 + 4 nb, fp16 hi part for even gid,
    // lo part for odd gid) at tokens 2 tig, 2 tig + 1 (first register) and 2 tig + 8, 2 tig + 9 (second); Z and S
    // of head gid / 2 + 4 nb are summed over those tokens (the odd lanes repeat the even lanes' sums)
    float zsum[NB], ssum[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) zsum[nb] = ssum[nb] = 0.f;
    const bool lo_part = gid & 1;
    constexpr int VSTR = RV_ ? 4 * 2 * RV_ * 4 : 0;  // records +4
    const uint32_t vstr = 4u * 2u * RV * 4u;
    // z/s words of tokens 2 tig, 2 tig + 1 (record (WT/2) pw + 8 mt + tig) and 2 tig + 8, 2 tig + 9 (+4 records)
    const uint32_t vzo = (uint32_t)DT * RK * 4u + (uint32_t)((WT / 2) * pw + tig) * 2u * RV * 4u;
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NS, slot = i & 1;
      const uint32_t sb = ring + (uint32_t)s * stage_bytes;
      // p of this stage comes from the key warp, usually later than the stage's records: sleep while waiting,
      // leaving the issue slots to the key warps
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&pF[pw][slot]), (uint32_t)((i >> 1) & 1), a.wait_ns, 128))) {
        s_abort = 1;
        break;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((i / NS) & 1), a.wait_ns))) {
        s_abort = 1;
        break;
      }
      const float* pb = reinterpret_cast<const float*>(pbase + slot * pbuf_bytes(NB));
      float2 pp[2][NB][2];
      float cacc[NB], czs[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int hh = (gid >> 1) + 4 * nb;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const float* row = pb + (mt * 4 * NB + hh) * PROW + 2 * tig;
          pp[mt][nb][0] = *reinterpret_cast<const float2*>(row);
          pp[mt][nb][1] = *reinterpret_cast<const float2*>(row + 8);
        }
        cacc[nb] = pb[PCORR / 4 + nb * 4 + tig];          // accumulator columns: head tig + 4 nb
        czs[nb] = pb[PCORR / 4 + nb * 4 + (gid >> 1)];    // this lane's Z, S: head gid / 2 + 4 nb
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&pE[pw][slot]));
      uint32_t zs[2][4];  // [m-tile][tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9]: z/s words
      {
        uint32_t t0w, t1w, t2w, t3w, t4w, t5w, t6w, t7w;
        lds_x4<VSTR>(sb + vzo, vstr, t0w, t2w, t4w, t6w);
        lds_x4<VSTR>(sb + vzo + 4u, vstr, t1w, t3w, t5w, t7w);
        zs[0][0] = t0w, zs[0][1] = t1w, zs[0][2] = t2w, zs[0][3] = t3w;
        zs[1][0] = t4w, zs[1][1] = t5w, zs[1][2] = t6w, zs[1][3] = t7w;
      }
      const int rb = i * DT + WT * pw;  // split-relative first token of this warp's 32
      const bool full_stage = (i + 1) * DT <= n_in;
      uint32_t bp[2][NB][2];
      float pz[NB], psw[NB];  // this stage's shares of Z and S (both m-tiles), folded in once below
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) pz[nb] = psw[nb] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        float zv[4], sv[4];
        bool val[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&zs[mt][k]));
          zv[k] = f.x;
          sv[k] = f.y;
          val[k] = full_stage || rb + 16 * mt + 2 * tig + (k & 1) + 8 * (k >> 1) < n_in;
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const float p4[4] = {pp[mt][nb][0].x, pp[mt][nb][0].y, pp[mt][nb][1].x, pp[mt][nb][1].y};
          __half hv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float wv = val[k] ? p4[k] * sv[k] : 0.f;
            pz[nb] += val[k] ? p4[k] * zv[k] : 0.f;
            psw[nb] += wv;
            const __half hi = __float2half_rn(wv);
            hv[k] = lo_part ? __float2half_rn(wv - __half2float(hi)) : hi;
          }
          bp[mt][nb][0] = pack_half2(hv[0], hv[1]);
          bp[mt][nb][1] = pack_half2(hv[2], hv[3]);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        zsum[nb] = fmaf(zsum[nb], czs[nb], pz[nb]);
        ssum[nb] = fmaf(ssum[nb], czs[nb], psw[nb]);
      }
      // accumulator columns 2 tig, 2 tig + 1 are head tig (+4 nb), fp16 hi and lo parts of W. The stage's 32-token
      // products are summed by the MMA from zero and folded into the running sums by round-to-nearest FMAs
      // (acc = acc corr + stage): accumulating inside the MMA across all stages would bias these sums of positive
      // terms by a rounding step per stage, which the near-cancellation of Z, S and M in the output magnifies.
#pragma unroll
      for (int mb = 0; mb < NBLK; ++mb) {
        // m-tile mt: records 8 mt + tig (tokens 2 tig, +1) and 8 mt + 4 + tig; channels gid (slot 0), gid + 8 (slot 1)
        uint32_t af[2][4];
        lds_x4<VSTR>(sb + (sd[mb][0] >> 5), vstr, af[0][0], af[0][2], af[1][0], af[1][2]);
        lds_x4<VSTR>(sb + (sd[mb][1] >> 5), vstr, af[0][1], af[0][3], af[1][1], af[1][3]);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          af[mt][0] = slot_f16x2(af[mt][0], sd[mb][0], sm[mb][0]);
          af[mt][1] = slot_f16x2(af[mt][1], sd[mb][1], sm[mb][1]);
          af[mt][2] = slot_f16x2(af[mt][2], sd[mb][0], sm[mb][0]);
          af[mt][3] = slot_f16x2(af[mt][3], sd[mb][1], sm[mb][1]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float tile[4];
          mma_f16_zero(tile, af[0], bp[0][nb][0], bp[0][nb][1]);
          mma_f16(tile, af[1], bp[1][nb][0], bp[1][nb][1]);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mb][nb][e] = fmaf(acc[mb][nb][e], cacc[nb], tile[e]);
        }
      }
      release_stage(i);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int h = tig + 4 * nb;
      if (h < g) {
        float* w = ws + (pw * 8 + h) * PSTR;
#pragma unroll
        for (int mb = 0; mb < NBLK; ++mb) {
          if (mb < nmb) {
            w[4 + mb * 16 + gid] = acc[mb][nb][0] + acc[mb][nb][1];
            w[4 + mb * 16 + gid + 8] = acc[mb][nb][2] + acc[mb][nb][3];
          }
        }
      }
      // Z and S of head gid / 2 + 4 nb: the four tig lanes of an even gid hold the 16 tokens' shares
      float zt = zsum[nb], st = ssum[nb];
      zt += __shfl_xor_sync(0xffffffffu, zt, 1);
      zt += __shfl_xor_sync(0xffffffffu, zt, 2);
      st += __shfl_xor_sync(0xffffffffu, st, 1);
      st += __shfl_xor_sync(0xffffffffu, st, 2);
      const int hh = (gid >> 1) + 4 * nb;
      if (hh < g && tig == 0 && !lo_part) {
        float* w = ws + (pw * 8 + hh) * PSTR;
        w[2] = zt;
        w[3] = st;
      }
    }
  }

  __syncthreads();
  float* part = a.part + ((size_t)bh * a.splits + split) * g * PSTR;
  if (s_abort) {  // drain the copies this CTA may still have in flight, then leave an empty partial
    if (tid == 0) {
      const int issued = s_issued;
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % NS]), (uint32_t)((i / NS) & 1), a.wait_ns);
    }
    for (int idx = tid; idx < g * PSTR; idx += DTHREADS) part[idx] = (idx % PSTR) == 0 ? -INFINITY : 0.f;
  } else {
    // ======== this split's partial (rotated basis): the warp pairs' sums weighted by 2^(m_w - max_w m_w) ========
    const int acols = 4 + nmb * 16;
    for (int idx = tid; idx < g * acols; idx += DTHREADS) {
      const int h = idx / acols, cidx = idx - h * acols;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < DW; ++w) M = fmaxf(M, ws[(w * 8 + h) * PSTR]);
      float val = M;
      if (cidx > 0) {
        val = 0.f;
#pragma unroll
        for (int w = 0; w < DW; ++w) {
          const float mw = ws[(w * 8 + h) * PSTR];
          const float e = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
          val = fmaf(e, ws[(w * 8 + h) * PSTR + cidx], val);
        }
      }
      part[h * PSTR + cidx] = val;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const bool last = atomicAdd(&a.cnt[bh], 1u) == (unsigned)(a.splits - 1);
    if (last) a.cnt[bh] = 0u;  // every split has arrived: the counter is ready for the next call
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ======== last CTA of (b, kh): weighted sum of the split partials, then the map to the original basis ========
  // T'_V arrives by one bulk copy while the partials arrive in chunks of splits; warp h (< g) keeps head h's running
  // maximum M_h and rescales with the weights e_s = 2^(m_s - M_h) (lanes over the chunk's splits); every thread
  // adds its items' sum e_s x_s (x: l, Z, S, M_j).
  float* Tsc = reinterpret_cast<float*>(smem);                     // [nzV][128]
  float* cp = reinterpret_cast<float*>(smem + L.chunks);           // chunk of split partials
  float* mrg = reinterpret_cast<float*>(smem + L.tail_reserve);    // merged partial [8][PSTR]
  float* escw = mrg + MAX_G * PSTR + 4 * MAX_G;                    // [MAX_SPLITS][8] weights of the chunk
  float* hst = escw + MAX_SPLITS * MAX_G;                          // rescale of the running sums [8]
  const float* pbp = a.part + (size_t)bh * a.splits * g * PSTR;
  const int S = a.splits;
  const uint32_t per_split = (uint32_t)g * PSTR * 4;
  const int chunk_splits = max(1, min(S, min((int)((L.tail_reserve - L.chunks) / per_split), MAX_SPLITS)));
  constexpr int ITEMS = (MAX_G * PSTR + DTHREADS - 1) / DTHREADS;
  constexpr int SPL = MAX_SPLITS / 32;  // splits per lane within a chunk
  const int icols = 4 + nzV;            // items of a head: m (unused), l, Z, S, M_0 .. M_(nzV - 1)
  float accI[ITEMS];
#pragma unroll
  for (int r = 0; r < ITEMS; ++r) accI[r] = 0.f;
  float M_run = -INFINITY;  // warp h's running maximum of head h
  uint32_t tphase = 0;
  fence_proxy_async_global();
  if (tid == 0 && nzV > 0) {  // T'_V on its own barrier
    fence_proxy_async_smem();
    mbar_expect_tx(smem_u32(&vbar_s), (uint32_t)nzV * D * 4);
    bulk_g2s(smem_u32(Tsc), TV.Tsc + so * D, (uint32_t)nzV * D * 4, smem_u32(&vbar_s));
  }
  for (int c0s = 0; c0s < S; c0s += chunk_splits) {
    const int n = min(chunk_splits, S - c0s);
    __syncthreads();  // previous chunk consumed
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_expect_tx(smem_u32(tbar), (uint32_t)n * per_split);
      bulk_g2s(smem_u32(cp), pbp + (size_t)c0s * g * PSTR, (uint32_t)n * per_split, smem_u32(tbar));
    }
    const bool okc = mbar_wait_bounded(smem_u32(tbar), tphase, a.wait_ns);
    if (!okc && tid == 0) mbar_wait_bounded(smem_u32(tbar), tphase, a.wait_ns);  // drain before leaving
    tphase ^= 1u;
    if (!__syncthreads_and(okc)) return;
    if (warp < g) {
      const int h = warp;
      float msp[SPL];
      float cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const int sp = lane + 32 * i;
        msp[i] = sp < n ? cp[(sp * g + h) * PSTR] : -INFINITY;
        cm = fmaxf(cm, msp[i]);
      }
      cm = warp_max(cm);
      const float Mn = fmaxf(M_run, cm);
      const float sc = (M_run == Mn) ? 1.f : exp2f(M_run - Mn);
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        const int sp = lane + 32 * i;
        if (sp < n) escw[sp * MAX_G + h] = msp[i] == -INFINITY ? 0.f : exp2f(msp[i] - Mn);
      }
      M_run = Mn;
      if (lane == 0) hst[h] = sc;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
      const int it = tid + r * DTHREADS;
      const int h = it / PSTR, col = it - h * PSTR;
      if (h < g && col >= 1 && col < icols) {
        float acc = accI[r] * hst[h];
        for (int sp = 0; sp < n; ++sp) acc = fmaf(escw[sp * MAX_G + h], cp[(sp * g + h) * PSTR + col], acc);
        accI[r] = acc;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < ITEMS; ++r) {
    const int it = tid + r * DTHREADS;
    const int h = it / PSTR, col = it - h * PSTR;
    if (h < g && col >= 1 && col < icols) mrg[h * PSTR + col] = accI[r];
  }
  bool okv = true;
  if (nzV > 0) okv = mbar_wait_bounded(smem_u32(&vbar_s), 0u, a.wait_ns);
  if (!okv && tid == 0) mbar_wait_bounded(smem_u32(&vbar_s), 0u, a.wait_ns);  // drain before leaving
  if (!__syncthreads_and(okv)) return;
  // the map to the original basis: wph warps per head, each over a range of the rotated channels, lane = four
  // original channels (a 128-bit segment of each T' row); the partial sums meet in shared memory
  constexpr int NWARPS = DTHREADS / 32;
  const int wph = max(1, NWARPS / g), h = warp / wph, qr = warp - h * wph;
  float4* rbuf = reinterpret_cast<float4*>(cp);  // [NWARPS][32] (the chunks are consumed)
  {
    float4 n = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < g) {
      const float* mh = mrg + h * PSTR;
      const int j0 = nzV * qr / wph, j1 = nzV * (qr + 1) / wph;
#pragma unroll 4
      for (int jj = j0; jj < j1; ++jj) {
        const float4 t = reinterpret_cast<const float4*>(Tsc + jj * D)[lane];
        const float aj = mh[4 + jj];
        n.x = fmaf(t.x, aj, n.x);
        n.y = fmaf(t.y, aj, n.y);
        n.z = fmaf(t.z, aj, n.z);
        n.w = fmaf(t.w, aj, n.w);
      }
    }
    rbuf[warp * 32 + lane] = n;
  }
  __syncthreads();
  if (h < g && qr == 0) {  // o_h[k] = base_k + (Z w_k - S w2_k + sum_j T'[j][k] M_j) / l
    const float* mh = mrg + h * PSTR;
    const float Lh = mh[1], zh = mh[2], sh = mh[3];
    const float4 w4 = reinterpret_cast<const float4*>(TV.wsum + so)[lane];
    const float4 v4 = reinterpret_cast<const float4*>(TV.wsum2 + so)[lane];
    const float4 b4 = reinterpret_cast<const float4*>(TV.base + so)[lane];
    float4 n = make_float4(fmaf(zh, w4.x, -sh * v4.x), fmaf(zh, w4.y, -sh * v4.y), fmaf(zh, w4.z, -sh * v4.z),
                           fmaf(zh, w4.w, -sh * v4.w));
    for (int q = 0; q < wph; ++q) {
      const float4 r = rbuf[(h * wph + q) * 32 + lane];
      n.x += r.x;
      n.y += r.y;
      n.z += r.z;
      n.w += r.w;
    }
    const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
    float4 o = make_float4(b4.x + n.x * inv, b4.y + n.y * inv, b4.z + n.z * inv, b4.w + n.w * inv);
    if (!(Lh > 0.f)) o = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(a.out + ((size_t)b * a.Hq + (size_t)kh * g + h) * D)[lane] = o;
  }
}

// splits per (sequence, KV head): one wave of CTAs (per_sm per SM) over the B * Hkv pairs, at most one per tile of
// the cache's capacity
static void split_plan(int B, int Hkv, int64_t T_cap, int device, int tile, int per_sm, int max_splits, int* splits,
                       int* chunk) {
  const long long bh = (long long)B * Hkv;
  const long long tiles = (T_cap + tile - 1) / tile;
  long long sp = std::max(1LL, (long long)per_sm * sm_count(device) / bh);
  sp = std::max(1LL, std::min(std::min(sp, tiles), (long long)max_splits));
  const long long ct = (tiles + sp - 1) / sp;
  *splits = (int)((tiles + ct - 1) / ct);
  *chunk = (int)(ct * tile);
}

DecodeLayout decode_layout(int B, int Hkv, int Hq, int64_t T_cap, int device) {
  DecodeLayout L{};
  const int g = Hq / Hkv;
  split_plan(B, Hkv, T_cap, device, dec_stage_tokens(g <= 4 ? 1 : 2), 1, MAX_SPLITS, &L.splits, &L.chunk);
  const size_t bh = (size_t)B * Hkv;
  size_t o = 0;
  L.off_cnt = o;
  o = align256(o + bh * sizeof(unsigned));
  L.off_part = o;
  o = align256(o + bh * (size_t)L.splits * g * PSTR * sizeof(float));
  L.total = o;
  return L;
}

template <int NB, int RK, int RV, int NBLK>
static cudaError_t launch_decode_kernel(cudaLaunchConfig_t& cfg, const ParamsDev& P, const DecArgs& a) {
  const cudaError_t e = ensure_dyn_smem((const void*)decode_kernel<NB, RK, RV, NBLK>, cfg.dynamicSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<NB, RK, RV, NBLK>, P, a);
}

// record lengths with a compile-time decode kernel: equal key and value budgets of 1.25 - 4 bits/element and the
// joint key/value splits of the Llama-shaped layer at 2.75, 2 and 1.33 bits/element
template <int NB, int NBLK>
static cudaError_t launch_decode_rw(cudaLaunchConfig_t& cfg, const ParamsDev& P, const DecArgs& a) {
  const int rk = P.t[0].r_words, rv = P.t[1].r_words;
#define KVTC_DECODE_RW(K, V) \
  if (rk == K && rv == V) return launch_decode_kernel<NB, K, V, NBLK>(cfg, P, a);
  KVTC_DECODE_RW(5, 5)
  KVTC_DECODE_RW(6, 4)
  KVTC_DECODE_RW(8, 8)
  KVTC_DECODE_RW(11, 11)
  KVTC_DECODE_RW(12, 12)
  KVTC_DECODE_RW(16, 16)
  KVTC_DECODE_RW(14, 8)
  KVTC_DECODE_RW(10, 6)
#undef KVTC_DECODE_RW
  return launch_decode_kernel<NB, 0, 0, NBLK>(cfg, P, a);
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
  const int nb = a.g <= 4 ? 1 : 2;
  a.stages = ring_stages_for(P.t[0].r_words, P.t[1].r_words, nb);
  a.scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int nblk = std::max(P.t[0].max_nz, P.t[1].max_nz) <= 64 ? 4 : 8;
  const size_t smem = decode_smem(P.t[0].r_words, P.t[1].r_words, a.stages, nb).total;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.splits, c.Hkv, B);
  cfg.blockDim = dim3(dec_threads(nb));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (nb == 1)
    e = nblk == 4 ? launch_decode_rw<1, 4>(cfg, P, a) : launch_decode_rw<1, 8>(cfg, P, a);
  else
    e = nblk == 4 ? launch_decode_rw<2, 4>(cfg, P, a) : launch_decode_rw<2, 8>(cfg, P, a);
  if (e != cudaSuccess) {
    set_error("decode_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return launch_check("decode_kernel");
}

}  // namespace kvtc
