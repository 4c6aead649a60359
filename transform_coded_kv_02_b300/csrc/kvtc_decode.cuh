// Decode over packed records: the split-K flash-decode kernel (with the q preparation in its prologue) and its
// launcher. kvtc_kernels.cu includes this header for the split plan and the dispatch; the kvtc_decode_part.cu
// units define KVTC_DECODE_KERNELS and compile the kernel's variants.
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
// Logits (base 2), per head h, token t, with Q_j = a log2(e) (T_K^-T q_h)_j sigma_j (T_K^-T = T_K for an orthogonal
// key transform; [NOVA-KV]'s key transform is not orthogonal) and w_j the slot width of channel
// j (b_j its code width; w_j = b_j except for a narrower channel sharing a key slot):
//   l_t = C0 + z_t C1 + s_t (sum_j Q_j 2^(w_j - b_j) A_tj - C2),  A_tj = 1 + c_tj 2^-w_j,
//   C0 = a log2(e) q.(T_K^-1 mu),  C1 = sum_{b_j>0} Q_j = a log2(e) q.w,  C2 = sum_{b_j>0} Q_j (2^(w_j - b_j) -
//   2^(-b_j - 1)) = a log2(e) q.w2  (w, w2: the key table's folded vectors),
// which is a log2(e) q.k^ for k^ = T_K^-1 y^, y^_j = mu_j + sigma_j (z + (c_j + 1/2) s 2^-b_j).
// Values, per head, with weights p_t (unnormalised softmax) and W_t = p_t s_t (value slots have w_j = b_j):
//   sum_t p_t y^_tj = l mu_j + sigma_j (Z - (1 - 2^(-b_j - 1)) S + M_j),  M_j = sum_t W_t A_tj,
//   Z = sum_t p_t z_t, S = sum_t W_t, l = sum_t p_t,
// so the original-basis sum is U_k = l (T_V^T mu)_k + Z w_k - S w2_k + sum_j T'_jk M_j with T'_jk = T_V[j][k]
// sigma_j, w_k = sum_j T'_jk, w2_k = sum_j T'_jk (1 - 2^(-b_j - 1)) (sums over b_j > 0), and o = U / l.
//
// Work split. A CTA owns one split (a token range) of one (sequence, KV head). Its warps are alike: each takes 32
// tokens of every ring stage (two 16-token MMA tiles), forms their logits (A = key codes, B = the heads' q'
// coefficients), runs the online softmax in the MMA's accumulator layout (a lane owns one head and four tokens),
// hands the weights W = p s to the value MMA's operand layout by warp shuffles, and accumulates M with A = value
// codes. At the end the warps' partials meet in shared memory, the CTA maps its merged sums to the original basis
// (U above), and the last CTA of the (sequence, head) to finish adds the splits' U with their softmax weights.
#pragma once
#include <type_traits>

namespace kvtc {

// ======================================================================================================
// decode over packed records
// ======================================================================================================
constexpr int PSTR = 132;              // floats per (warp or split, head) partial: m, l, Z, S | U or M [128]
constexpr int WTOK = 32;               // tokens of one warp per ring stage
constexpr int RING_BUDGET = 160 * 1024;
constexpr int MAX_STAGES = 8;
constexpr int MAX_SPLITS = 256;
constexpr int HC = 4;                  // per-head constants: C0, C1, C2, 2^-e

// Warps per CTA (nw): sixteen for one 8-column block of heads when two stages of 512 tokens fit the ring (more
// than four 16-channel blocks then keep their slot descriptors and q' operands in shared memory, so that a thread
// fits 128 registers), eight otherwise.
__host__ __device__ constexpr bool dec_desc_smem(int nw, int nblk) { return nw == 16 && nblk > 4; }
__host__ __device__ constexpr int dec_stage_tokens(int nw) { return WTOK * nw; }

struct DecArgs {
  CacheView c;              // the records (dense or paged) and the parameter set of each (z, KV head)
  const __nv_bfloat16* q;   // [B][Hq][128]
  const int32_t* seq_lens;  // [c.B]
  const int32_t* q_pos;     // [c.B] query positions for the rotary embedding, or null
  unsigned* cnt;    // [B*Hkv] arrival counters: zero before a call, left at zero after it
  float* part;      // [B*Hkv][splits][g][PSTR] split partials (m, l, -, -, U[128])
  float* out;       // [B][Hq][128]
  long long wait_ns;
  int B, Hkv, Hq, g, splits, stages;  // B: virtual sequences z of the launch (layers x sequences)
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

struct DecSmem {  // byte offsets into the dynamic shared memory of decode_kernel
  uint32_t stage_bytes, qa, hc, tab, pro, tsl, total;
};
// slot descriptor tables: keys [8 blocks][4 tig][2 slots] and values [8 blocks][8 gid][2 slots] of (descriptor,
// mask), then the logit MMA's B fragments per lane [8 blocks][32 lanes] (two words), then the pair (keys, [8][4][2])
// and channel (values, [8][8][2]) at each position of the decode's lane order
constexpr uint32_t TAB_BYTES = (8u * 4u * 2u + 8u * 8u * 2u) * 8u + 8u * 32u * 8u + 64u + 128u;
constexpr uint32_t SMEM_LIMIT = 227u * 1024u;   // dynamic shared memory a CTA may hold
constexpr uint32_t SMEM_STATIC = 1024u;         // room left for the kernel's static shared variables

// Epilogue scratch (floats) in the ring's bytes once the ring is consumed: the warps' partials [NW][8][PSTR], the
// CTA's merged partial [8][PSTR], the splits' merged M [8][128], the heads' merged l, Z, S [8][4], the splits'
// weights [MAX_SPLITS][8], the row blocks' partial dot products [NT / KW][8][KW] and a chunk of split partials
// [MERGE_CHUNK] (global merge); the last CTA of the global merge stages
// T'_V [128][128] and T_V^T mu, w, w2 [3][128] at the start (over the warps' partials, dead by then).
constexpr uint32_t MERGE_CHUNK = 12288;  // floats of split partials the global merge stages at once
struct DecEpi {
  uint32_t wpart, mrg, mg, hs, esw, rot, chunk, tfull, end;
};
// chunk: room for the global merge's staged partials (the workspace path only)
__host__ __device__ inline DecEpi decode_epi(int nw, int nt, bool chunk) {
  DecEpi e;
  e.wpart = 0;
  e.tfull = 0;
  e.mrg = e.wpart + (uint32_t)nw * MAX_G * PSTR;
  e.mg = e.mrg + MAX_G * PSTR;
  e.hs = e.mg + MAX_G * D;
  e.esw = e.hs + MAX_G * 4;
  e.rot = e.esw + MAX_SPLITS * MAX_G;
  e.chunk = e.rot + (uint32_t)MAX_G * nt;
  e.end = e.chunk + (chunk ? MERGE_CHUNK : 0u);
  const uint32_t tend = (uint32_t)(D + 3) * D;  // T'_V rows and the three column vectors
  if (e.mrg < tend) {                           // keep the merge scratch clear of the staged T'_V
    const uint32_t sh = tend - e.mrg;
    e.mrg += sh, e.mg += sh, e.hs += sh, e.esw += sh, e.rot += sh, e.chunk += sh, e.end += sh;
  }
  return e;
}

// [0, qa): the ring of record stages, then the epilogue scratch above | qa: q' operands [16 columns][128] fp16 |
// hc: per-head constants [8][HC] | tab: slot descriptor tables | pro: prologue scratch (q [8][128], partial q~ [QPARTS][8][128], coefficient
// scales [8]) | tsl (cluster merge, cs > 0): this CTA's columns of T'_V [128][128 / cs] and of T_V^T mu, w, w2
// [3][128 / cs]
__host__ __device__ inline DecSmem decode_smem(int RK, int RV, int stages, int nw, int cs) {
  DecSmem s;
  const int nt = 32 * nw, parts = nt / D;
  s.stage_bytes = (uint32_t)dec_stage_tokens(nw) * (RK + RV) * 4u;
  const uint32_t ring = (uint32_t)stages * s.stage_bytes;
  const uint32_t epi = decode_epi(nw, nt, cs == 0).end * 4u;
  const uint32_t r = ring > epi ? ring : epi;
  s.qa = align128u(r);
  s.hc = s.qa + 16u * D * 2u;
  s.tab = align128u(s.hc + MAX_G * HC * 4u);
  s.pro = align128u(s.tab + TAB_BYTES);
  s.tsl = align128u(s.pro + (uint32_t)(MAX_G * D + parts * MAX_G * D + MAX_G) * 4u);
  s.total = s.tsl + (cs > 0 ? (uint32_t)(D + 3) * (D / cs) * 4u : 0u);
  return s;
}

// ring stages: as many as RING_BUDGET (and the CTA's shared memory left beside the other regions) holds, 2 to 8
__host__ __device__ inline int ring_stages_for(int RK, int RV, int nw, int cs) {
  const DecSmem z = decode_smem(RK, RV, 0, nw, cs);
  const uint32_t other = z.total - z.qa;
  uint32_t budget = SMEM_LIMIT - SMEM_STATIC - other;
  budget = budget < (uint32_t)RING_BUDGET ? budget : (uint32_t)RING_BUDGET;
  const int n = (int)(budget / z.stage_bytes);
  return n > MAX_STAGES ? MAX_STAGES : (n < 2 ? 2 : n);
}

// The map of merged rotated-basis sums to the original basis for output columns [k0, k0 + KW) of every head:
// o_k = (l base_k + Z w_k - S w2_k + sum_j T'[j][k] M_j) / l, with tsl = T' columns [128][KW], bsl = base, w, w2
// columns [3][KW], mg = merged M [8][128] (16-byte aligned, zero past nzV up to a multiple of four), hs = merged
// (l, Z, S) [8][4]. Thread (row block, column) sums its rows for every head (one T' element serves all heads, one
// 16-byte load four rows of M); rot [NT / KW][8][KW] gathers the row blocks' sums.
template <int NT>
__device__ __forceinline__ void rotate_out(const float* tsl, const float* bsl, const float* mg, const float* hs,
                                           float* rot, int g, int KW, int k0, int nzV, float* outp) {
  const int tid = threadIdx.x;
  const int JP = NT / KW, kl = tid % KW, jp = tid / KW;
  const int n4 = (nzV + 3) >> 2;  // groups of four rows (rows past nzV are zero in T' and in mg)
  const int q0 = n4 * jp / JP, q1 = n4 * (jp + 1) / JP;
  float acc[MAX_G];
#pragma unroll
  for (int h = 0; h < MAX_G; ++h) acc[h] = 0.f;
  for (int q = q0; q < q1; ++q) {
    const int j = 4 * q;
    float t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) t[u] = tsl[(j + u) * KW + kl];
#pragma unroll
    for (int h = 0; h < MAX_G; ++h)
      if (h < g) {
        const float4 m = *reinterpret_cast<const float4*>(mg + h * D + j);
        acc[h] = fmaf(t[0], m.x, fmaf(t[1], m.y, fmaf(t[2], m.z, fmaf(t[3], m.w, acc[h]))));
      }
  }
#pragma unroll
  for (int h = 0; h < MAX_G; ++h)
    if (h < g) rot[(jp * MAX_G + h) * KW + kl] = acc[h];
  __syncthreads();
  for (int o = tid; o < g * KW; o += NT) {
    const int h = o / KW, c = o - h * KW;
    float sacc = 0.f;
    for (int p = 0; p < JP; ++p) sacc += rot[(p * MAX_G + h) * KW + c];
    const float l = hs[h * 4];
    const float u = fmaf(l, bsl[c], fmaf(hs[h * 4 + 1], bsl[KW + c], fmaf(-hs[h * 4 + 2], bsl[2 * KW + c], sacc)));
    outp[h * D + k0 + c] = l > 0.f ? u / l : 0.f;
  }
}

// The cluster's merged M_j = sum_r e_r M_rj over its CSX splits (distributed shared memory): every thread's loads
// for all its items and ranks are issued before the first is used (the item index clamped, so that none is
// predicated).
template <int CSX, int NT>
__device__ __forceinline__ void cluster_merge_m(uint32_t mrg_a, const float* esw, float* mg, int g, int nzV) {
  constexpr int IT = (MAX_G * D + NT - 1) / NT;
  const int n = g * nzV;
  if (n == 0) return;
  float v[IT][CSX];
  int hj[IT];
#pragma unroll
  for (int r = 0; r < IT; ++r) {
    const int idx = min((int)threadIdx.x + NT * r, n - 1);
    const int h = idx / nzV, j = idx - h * nzV;
    hj[r] = h * D + j;
    const uint32_t la = mrg_a + (uint32_t)(h * PSTR + 4 + j) * 4u;
#pragma unroll
    for (int c = 0; c < CSX; ++c) v[r][c] = ld_dsmem(dsmem_addr(la, c));
  }
#pragma unroll
  for (int r = 0; r < IT; ++r) {
    if ((int)threadIdx.x + NT * r < n) {
      const int h = hj[r] / D;
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CSX; ++c) acc = fmaf(esw[c * MAX_G + h], v[r][c], acc);
      mg[hj[r]] = acc;
    }
  }
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
// NB: 8-column blocks of the logit MMA's n dimension (4 heads each, fp16 hi and lo columns). NBLK: 16-channel
// blocks processed per tensor (blocks past a set's last nonzero-width channel hold zero masks and coefficients).
// CL: the splits of a (sequence, head) form one thread-block cluster (gridDim.x = cluster size) and merge through
// distributed shared memory; otherwise they merge through the workspace, the last to arrive doing the merge.
// SW bit 0 (keys) / bit 1 (values): every channel block the decode reads, in every set, has both slots of each
// lane in one code word (the table's single_word flags): one shared load per block and no per-block test.
template <int NB, int RK_, int RV_, int NBLK, bool CL, int NW, int SW>
__global__ void __launch_bounds__(32 * NW, 1) decode_kernel(ParamsDev P, DecArgs a) {
  constexpr int NT = 32 * NW, ST = WTOK * NW;
  constexpr int QPARTS = NT / D, KQ = D / QPARTS;  // q preparation: threads per channel, k's per thread
  extern __shared__ __align__(128) uint8_t smem[];
  // barriers live outside the dynamic region, which the epilogue reuses wholesale
  __shared__ __align__(8) uint64_t full[MAX_STAGES];
  __shared__ unsigned rel[MAX_STAGES];  // warps done with the stage in each ring slot
  __shared__ int s_abort, s_last, s_issued;
  __shared__ long long s_trange[2];  // the split's token range, for the refills (kept out of the loop's registers)
  const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;  // b: virtual sequence (layer, sequence)
  const int bh = b * a.Hkv + kh;
  const int set = view_set(a.c, b, kh);
  const int bseq = b % a.c.B;  // the sequence within its layer
  const TensorDev& TK = P.t[0];
  const TensorDev& TV = P.t[1];
  const int RK = RK_ ? RK_ : TK.r_words, RV = RV_ ? RV_ : TV.r_words;
  const int NS = a.stages, g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const size_t so = (size_t)set * D;
  const int CS = CL ? a.splits : 0;  // cluster size
  const DecSmem L = decode_smem(RK, RV, NS, NW, CS);
  const uint32_t stage_bytes = L.stage_bytes;
  __half* qa = reinterpret_cast<__half*>(smem + L.qa);  // [16 columns][128 channels]
  float* hc = reinterpret_cast<float*>(smem + L.hc);    // [8 heads][HC]

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      rel[s] = 0u;
    }
    fence_mbar_init();
    s_abort = 0;
    s_issued = 0;
  }
  // ---- parameters only (nothing a previous kernel writes): one round of loads, left in flight while the kernel
  // waits for its predecessor and fetches q ----
  // key slots: pair 8 kb + 4 i + tig of token rows 32 warp + gid (+ 8, 16, 24); value slots: channel 16 mb + 8 i +
  // gid of the two-token records 16 warp + tig (+ 4, 8, 12)
  const int nzK = __ldg(TK.nz + set), nzV = __ldg(TV.nz + set);
  constexpr bool DS = dec_desc_smem(NW, NBLK);
  constexpr int NR = DS ? 1 : NBLK;  // blocks whose descriptors and q' operands live in registers
  uint32_t kd[NR][2], km[NR][2], vd[NR][2], vm[NR][2];  // raw slot entries first, descriptors later
  // slot descriptors in the decode's lane order (keys [8][4 tig][2], values [8][8 gid][2]): a lane's two slots of a
  // channel block sit in one code word wherever the layout allowed it; `single` marks the blocks where every lane's
  // two slots do (one shared load serves both)
  const uint32_t* kslp = TK.slp + (size_t)set * 64;
  const uint32_t* vslp = TV.slp + (size_t)set * 128;
  const uint32_t smask = __ldg(TK.single + set);
  uint32_t rawk = 0u, rawv = 0u;  // DS: the table entry this thread fills
  if constexpr (DS) {
    if (tid < NBLK * 8) rawk = __ldg(kslp + tid);
    if (tid < NBLK * 16) rawv = __ldg(vslp + tid);
  } else {
#pragma unroll
    for (int kb = 0; kb < NBLK; ++kb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        kd[kb][i] = __ldg(kslp + (kb * 4 + tig) * 2 + i);
        vd[kb][i] = __ldg(vslp + (kb * 8 + gid) * 2 + i);
      }
  }
  // the pair (keys) and channel (values) at each position, for the q' operands and the value sums' write-back
  uint32_t rawidx = 0u;
  if (tid < 48)
    rawidx = __ldg(reinterpret_cast<const uint32_t*>(tid < 16 ? TK.idx + (size_t)set * 64 : TV.idx + (size_t)set * 128) +
                   (tid < 16 ? tid : tid - 16));
  if constexpr (CL) {  // this CTA's output columns of T'_V and of T_V^T mu, w, w2, copied while the CTA works
    const int KW = D / CS, k0 = split * KW, cpr = KW / 4;  // 16-byte chunks per row
    const uint32_t tdst = smem_u32(smem + L.tsl);
    for (int c = tid; c < (D + 3) * cpr; c += NT) {
      const int row = c / cpr, cc = c - row * cpr;
      const float* src = row < D ? TV.Tsc + (so + row) * D : (row == D ? TV.base : row == D + 1 ? TV.wsum : TV.wsum2) + so;
      cp_async16(tdst + (uint32_t)(row * KW + 4 * cc) * 4u, src + k0 + 4 * cc);
    }
    cp_async_commit();
  }
  // q preparation: this thread's slice of T^-1 (T^T for an orthogonal T; rows KQ part .. KQ part + KQ - 1,
  // column j), channel j's sigma and widths; warp h < 8: the folded key vectors at its lane's four entries
  const int qj = tid & (D - 1), qpart = tid / D;
  float tt[KQ];
  {
    const float* TTc = TK.Tq + so * D + (size_t)(KQ * qpart) * D + qj;  // q~ = T_K^-T q
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
  // rotary embedding of q: warp h's copy of the 64 frequencies (turns), by asynchronous copies into the prologue's
  // partial-q~ scratch, which the q preparation writes only after the embedding has read them
  unsigned long long* const rturn =
      reinterpret_cast<unsigned long long*>(smem + L.pro + (uint32_t)(MAX_G * D) * 4u) + warp * (D / 2);
  if (a.q_pos && warp < g) {
    cp_async16(smem_u32(rturn + 2 * lane), P.rope_turns + 2 * lane);
    cp_async_commit();
  }
  __syncthreads();

  // The previous kernel of the stream (an append, say) may still be running: q, the lengths and the records are
  // read only after it has completed.
  pdl_wait();
  // q and the length first, so that their loads do not queue behind the ring's copies
  uint2 qraw = make_uint2(0u, 0u);
  if (warp < g) qraw = reinterpret_cast<const uint2*>(a.q + ((size_t)b * a.Hq + (size_t)kh * g + warp) * D)[lane];
  const long long Lseq = max(0LL, min((long long)a.seq_lens[bseq], a.c.T_cap));
  const long long qpos = a.q_pos ? (long long)a.q_pos[bseq] : 0LL;

  // this sequence's tokens spread over all the splits in whole warp blocks, sized from its own length, so that a
  // short sequence in a long cache (or in a ragged batch) keeps every split busy
  const long long chunk = ((Lseq + a.splits - 1) / a.splits + WTOK - 1) / WTOK * WTOK;
  const long long t0 = min((long long)split * chunk, Lseq);
  const long long t1 = min(t0 + chunk, Lseq);
  const int n_in = (int)(t1 - t0);
  const int ntiles = (n_in + ST - 1) / ST;

  // ---- record stages stream into the ring by bulk copies: thread 0 fills the ring, then the last of the NW warps
  // to release a slot refills it at once with the stage NS further on ----
  const uint32_t ring = smem_u32(smem);
  // stage i of the split's token range [ta, tz)
  auto issue_tile = [&](int i, long long ta, long long tz) {
    const int s = i % NS;
    const long long tb = ta + (long long)i * ST;
    long long n = min((long long)ST, tz - tb);
    n = min((n + 3) & ~3LL, a.c.T_cap - tb);
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t dst = ring + (uint32_t)s * stage_bytes;
    if (a.c.bt == nullptr) {
      const uint32_t* krec = a.c.rec[0] + (size_t)bh * a.c.T_cap * RK;
      const uint32_t* vrec = a.c.rec[1] + (size_t)bh * a.c.T_cap * RV;  // two-token records: same bytes per token
      const uint32_t kbytes = (uint32_t)(n * RK * 4), vbytes = (uint32_t)(n * RV * 4);
      mbar_expect_tx(bar, kbytes + vbytes);
      bulk_g2s(dst, krec + tb * RK, kbytes, bar);
      bulk_g2s(dst + ST * RK * 4, vrec + tb * RV, vbytes, bar);
      return;
    }
    // paged: one copy per tensor and page the stage touches (pages start at multiples of 32 tokens, so every
    // piece starts and ends on a 16-byte boundary); the barrier expects the bytes of the pages in range, and a
    // page index out of range is reported and its tokens left as they are. Positions fit 32 bits (checked by the
    // host) and pages hold a power of two of tokens.
    const int psh = a.c.P_shift, p0 = (int)tb, p1 = (int)(tb + n);
    const int32_t* btr = a.c.bt + (size_t)b * a.c.max_pages;
    uint32_t bytes = 0;
    for (int p = p0; p < p1;) {
      const int e = min(p1, ((p >> psh) + 1) << psh);
      const unsigned pg = (unsigned)__ldg(btr + (p >> psh));
      if (pg < (unsigned long long)a.c.n_pages) bytes += (uint32_t)(e - p) * (uint32_t)(RK + RV) * 4u;
      p = e;
    }
    mbar_expect_tx(bar, bytes);
    for (int p = p0; p < p1;) {
      const int e = min(p1, ((p >> psh) + 1) << psh);
      const unsigned pg = (unsigned)__ldg(btr + (p >> psh));
      if (pg < (unsigned long long)a.c.n_pages) {
        const uint32_t cnt = (uint32_t)(e - p), o = (uint32_t)(p - p0);
        // token row within the pool
        const size_t row = (((size_t)pg * a.Hkv + kh) << psh) + (size_t)(p & ((1 << psh) - 1));
        bulk_g2s(dst + o * RK * 4u, a.c.rec[0] + row * RK, cnt * RK * 4u, bar);
        bulk_g2s(dst + ST * RK * 4 + o * RV * 4u, a.c.rec[1] + row * RV, cnt * RV * 4u, bar);
      } else {
        atomicOr(&g_status, ST_BAD_INDEX);
      }
      p = e;
    }
  };
  // this warp is done reading stage i: the last warp to say so issues stage i + NS into the same slot (its
  // acquire-release count orders every warp's reads of the slot before the refill's writes)
  auto release_stage = [&](int i) {
    __syncwarp();
    if (lane == 0) {
      const int s = i % NS;
      unsigned old;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(&rel[s])) : "memory");
      if (old == (unsigned)NW - 1u) {
        rel[s] = 0u;
        if (i + NS < ntiles) {
          fence_proxy_async_smem();
          issue_tile(i + NS, s_trange[0], s_trange[1]);
          atomicMax(&s_issued, i + NS + 1);
        }
      }
    }
  };
  // The last warp fills the ring, a stage per lane, while the q preparation runs. With sixteen warps (512-token
  // stages, a few per split) it issues only the first 48 KB of stages now (at least one) and the rest just before
  // the main loop: every CTA's first stage then shares the memory system with fewer of the other CTAs' later stages,
  // and arrives sooner (32768-token Llama layer, one 45 KB stage first: 26.6 -> 24.6 us; 131072 tokens at 1.33 bits,
  // two 20 KB stages first: 44.9 -> 41.9 us). Eight-warp kernels, with deeper rings of shorter stages, fill the
  // whole ring at once.
  constexpr bool DEFER = NW == 16;
  const int first = DEFER ? max(1, min(NS, (int)((48u * 1024u) / stage_bytes))) : NS;
  if (warp == NW - 1) {
    if (lane < first && lane < ntiles) issue_tile(lane, t0, t1);
    if (lane == 0) {
      s_trange[0] = t0;
      s_trange[1] = t1;
      if (!CL && split == 0 && nzV > 0)  // the merging split reads the scaled T_V rows at its end
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(TV.Tsc + so * D), "r"((uint32_t)nzV * D * 4)
                     : "memory");
      s_issued = min(first, ntiles);
    }
  }
  // slot descriptors (blocks past the set's last nonzero-width channel get zero masks)
  const int nkb = (nzK + 15) >> 4, nmb = (nzV + 15) >> 4;
  // byte offsets of this lane's key token row (gid of the warp's block) and value record (tig) in a stage
  const uint32_t krow = (uint32_t)(WTOK * warp + gid) * RK * 4u;
  const uint32_t vrow = (uint32_t)ST * RK * 4u + (uint32_t)((WTOK / 2) * warp + tig) * 2u * RV * 4u;
  uint2* const ktab = reinterpret_cast<uint2*>(smem + L.tab);  // [NBLK][4 tig][2 slots]: descriptor, mask
  uint2* const vtab = ktab + 8 * 4 * 2;                         // [NBLK][8 gid][2 slots]
  uint2* const qfrag = vtab + 8 * 8 * 2;                        // [NBLK][32 lanes]: logit B fragments
  uint32_t* const kidx32 = reinterpret_cast<uint32_t*>(qfrag + 8 * 32);  // [8][4][2] pair indices (bytes)
  const uint8_t* const kidx = reinterpret_cast<const uint8_t*>(kidx32);
  const uint8_t* const vidx = kidx + 64;                                  // [8][8][2] channel indices
  if (tid < 48) kidx32[tid] = rawidx;
  if constexpr (DS) {  // record-relative descriptors; the lanes add their row offsets
    if (tid < NBLK * 8) {  // key position (block tid / 8, lane (tid / 2) % 4, slot tid % 2)
      const uint32_t dk = (tid >> 3) < nkb ? rawk : 0u;
      const uint32_t b0 = (dk >> 16) & 255u, b1 = dk >> 24, w = b0 > b1 ? b0 : b1;
      uint2 e;
      slot_decode_desc(4u * (1u + (dk & 255u)), (dk >> 8) & 255u, w, b0, b1, e.x, e.y);
      ktab[tid] = e;
    }
    if (tid < NBLK * 16) {  // value position (block tid / 16, lane (tid / 2) % 8, slot tid % 2)
      const uint32_t dv = (tid >> 4) < nmb ? rawv : 0u;
      const uint32_t bw = (dv >> 16) & 255u;
      uint2 e;
      slot_decode_desc(4u * (2u + (dv & 255u)), (dv >> 8) & 255u, bw, bw, bw, e.x, e.y);
      vtab[tid] = e;
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < NBLK; ++kb)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t dk = kb < nkb ? kd[kb][i] : 0u;
        const uint32_t b0 = (dk >> 16) & 255u, b1 = dk >> 24, w = b0 > b1 ? b0 : b1;
        slot_decode_desc(krow + 4u * (1u + (dk & 255u)), (dk >> 8) & 255u, w, b0, b1, kd[kb][i], km[kb][i]);
        const uint32_t dv = kb < nmb ? vd[kb][i] : 0u;
        const uint32_t bw = (dv >> 16) & 255u;
        slot_decode_desc(vrow + 4u * (2u + (dv & 255u)), (dv >> 8) & 255u, bw, bw, bw, vd[kb][i], vm[kb][i]);
      }
  }

  // ---- q preparation: per-head constants from dot products of q with the folded vectors, then
  // q~ = T_K q and the MMA coefficients Q_j 2^(w_j - b_j) 2^e_h as fp16 hi + lo pairs ----
  {
    float* qs = reinterpret_cast<float*>(smem + L.pro);  // [8][128]
    float* red = qs + MAX_G * D;                          // [QPARTS][8][128]
    float* esc = red + QPARTS * MAX_G * D;                // [8] 2^e_h
    if (warp >= g && warp < MAX_G && lane == 0) {  // columns of no head: zero coefficients, unit scale
      hc[warp * HC + 0] = hc[warp * HC + 1] = hc[warp * HC + 2] = 0.f;
      hc[warp * HC + 3] = 1.f;
      esc[warp] = 1.f;
    }
    if (warp < g) {  // warp h: head h's row of q, its norm and its three dot products
      const int h = warp;
      float4 qv = make_float4(bf16_bits_f(qraw.x & 0xFFFFu), bf16_bits_f(qraw.x >> 16),
                              bf16_bits_f(qraw.y & 0xFFFFu), bf16_bits_f(qraw.y >> 16));
      if (a.q_pos) {  // rotary embedding at the query's position: pairs (e, e + 64) sit in lanes l and l ^ 16
        cp_async_wait_all();
        __syncwarp();
        float* v = reinterpret_cast<float*>(&qv);
        const float sg = lane < 16 ? -1.f : 1.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // the angle in turns, reduced exactly (64-bit fixed point, wrapping), as a signed fraction in [-1/2, 1/2)
          const unsigned long long fr = rturn[(4 * lane + u) & (D / 2 - 1)];
          const long long tw = (long long)((unsigned long long)qpos * fr);
          float sn, cs;
          sincospif((float)tw * 0x1p-63f, &sn, &cs);
          const float pv = __shfl_xor_sync(0xffffffffu, v[u], 16);
          v[u] = fmaf(sg * pv, sn, v[u] * cs);
        }
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
      if (h < g) {
        float acc0 = 0.f, acc1 = 0.f;
        const float4* q4 = reinterpret_cast<const float4*>(qs + h * D + KQ * qpart);
#pragma unroll
        for (int k4 = 0; k4 < KQ / 4; ++k4) {
          const float4 v = q4[k4];
          acc0 = fmaf(tt[4 * k4], v.x, acc0);
          acc1 = fmaf(tt[4 * k4 + 1], v.y, acc1);
          acc0 = fmaf(tt[4 * k4 + 2], v.z, acc0);
          acc1 = fmaf(tt[4 * k4 + 3], v.w, acc1);
        }
        red[(qpart * MAX_G + h) * D + qj] = acc0 + acc1;
      }
    }
    __syncthreads();
    if (tid < D) {
      const int j = qj, bj = q_bj, wj = q_bj > q_bp ? q_bj : q_bp;  // slot width of the channel pair
      const float f = bj > 0 ? a.scale_log2 * q_sg * exp2i(wj - bj) : 0.f;
#pragma unroll
      for (int h = 0; h < MAX_G; ++h) {
        float c = 0.f;
        if (h < g) {
          float qt = 0.f;
#pragma unroll
          for (int p = 0; p < QPARTS; ++p) qt += red[(p * MAX_G + h) * D + j];
          c = qt * f * esc[h];
        }
        const __half hi = __float2half_rn(c);
        const __half lo = __float2half_rn(c - __half2float(hi));
        qa[(2 * h) * D + j] = hi;
        qa[(2 * h + 1) * D + j] = lo;
      }
    }
    __syncthreads();
    if constexpr (DS) {  // each lane's B fragments of every channel block, one 8-byte row per lane
      if (tid < NBLK * 32) {  // slot i of lane t: the channel pair kidx[kb][t][i]
        const int kb = tid >> 5, ln = tid & 31, col = ln >> 2, t = ln & 3;
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qa);
        qfrag[tid] = make_uint2(q32[col * (D / 2) + kidx[(kb * 4 + t) * 2]], q32[col * (D / 2) + kidx[(kb * 4 + t) * 2 + 1]]);
      }
      __syncthreads();
    }
  }

  // ============ main loop: warp w owns tokens [32 w, 32 w + 32) of every stage ============
  // B operand of the logit MMA: coefficients, k = channels 16 kb + 2 tig (+1, +8, +9), n = column gid (head
  // gid / 2 + 4 nb, fp16 hi part for even gid, lo part for odd gid)
  const uint32_t* qa32 = reinterpret_cast<const uint32_t*>(qa);
  uint32_t qb[NR][NB][2];  // (DS: read from qa at each use)
  if constexpr (!DS) {
#pragma unroll
    for (int kb = 0; kb < NBLK; ++kb)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int col = nb * 8 + gid;
        qb[kb][nb][0] = qa32[col * (D / 2) + kidx[(kb * 4 + tig) * 2]];
        qb[kb][nb][1] = qa32[col * (D / 2) + kidx[(kb * 4 + tig) * 2 + 1]];
      }
  }
  // this lane's softmax head in column block nb: tig + 4 nb, over the tokens 32 w + gid + 8 m (m = 0..3)
  float C0[NB], C1[NB], C2[NB], qsc[NB], m_run[NB], l_run[NB], zsum[NB], ssum[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int h = tig + 4 * nb;
    C0[nb] = hc[h * HC + 0];
    C1[nb] = hc[h * HC + 1];
    C2[nb] = hc[h * HC + 2];
    qsc[nb] = hc[h * HC + 3];
    m_run[nb] = -INFINITY;
    l_run[nb] = zsum[nb] = ssum[nb] = 0.f;
  }
  // value sums M: channels 16 mb + gid (+8) x columns 2 tig, 2 tig + 1 (head tig + 4 nb, fp16 hi and lo parts of W)
  float vacc[NBLK][NB][4];
#pragma unroll
  for (int mb = 0; mb < NBLK; ++mb)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) vacc[mb][nb][0] = vacc[mb][nb][1] = vacc[mb][nb][2] = vacc[mb][nb][3] = 0.f;
  // the value MMA's B operand: this lane holds column gid at tile tokens 2 tig, 2 tig + 1 (+8), which the logit
  // layout keeps in lanes (2 tig) * 4 + gid / 2 and (2 tig + 1) * 4 + gid / 2, one packed (hi, lo) word per token
  const int srcA = 8 * tig + (gid >> 1), srcB = srcA + 4;
  const uint32_t psel = (gid & 1) ? 0x7632u : 0x5410u;
  const uint32_t kzo = (uint32_t)(WTOK * warp + gid) * RK * 4u;  // key z/s word of token row gid
  // value z/s word of token gid: record (gid / 2) of the warp's 16, word gid & 1
  const uint32_t vzo = (uint32_t)ST * RK * 4u + (uint32_t)((WTOK / 2) * warp + (gid >> 1)) * 2u * RV * 4u +
                       4u * (uint32_t)(gid & 1);
  constexpr int KSTR = RK_ ? 8 * RK_ * 4 : 0;       // token rows +8
  constexpr int VSTR = RV_ ? 4 * 2 * RV_ * 4 : 0;   // records +4
  const uint32_t kstr = 8u * RK * 4u, vstr = 4u * 2u * RV * 4u;

  if (DEFER && warp == NW - 1) {  // the rest of the ring, a stage per lane
    if (lane >= first && lane < NS && lane < ntiles) issue_tile(lane, t0, t1);
    if (lane == 0) atomicMax(&s_issued, min(NS, ntiles));
  }
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % NS;
    const uint32_t sb = ring + (uint32_t)s * stage_bytes;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((i / NS) & 1), a.wait_ns))) {
      s_abort = 1;
      break;
    }
    const int r0 = i * ST + WTOK * warp;  // split-relative first token of this warp's block
    if (r0 >= n_in) {                     // past the split's end (its last stage only)
      release_stage(i);
      continue;
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
      if (kb >= nkb) break;  // blocks past the set's last nonzero-width key channel (the same for the whole CTA)
      uint32_t d0, m0, d1, m1, a0, a1;  // the two slots' descriptors, masks and stage addresses
      if constexpr (DS) {
        const uint4 e = reinterpret_cast<const uint4*>(ktab)[kb * 4 + tig];
        d0 = e.x, m0 = e.y, d1 = e.z, m1 = e.w;
        a0 = sb + krow + (d0 >> 5), a1 = sb + krow + (d1 >> 5);
      } else {
        d0 = kd[kb][0], m0 = km[kb][0], d1 = kd[kb][1], m1 = km[kb][1];
        a0 = sb + (d0 >> 5), a1 = sb + (d1 >> 5);
      }
      uint32_t af[2][4];  // rows gid, gid + 8 (m-tile 0), gid + 16, gid + 24 (m-tile 1)
      lds_x4<KSTR>(a0, kstr, af[0][0], af[0][1], af[1][0], af[1][1]);
      if ((SW & 1) || ((smask >> kb) & 1u)) {  // both slots in the word just loaded
        af[0][2] = af[0][0], af[0][3] = af[0][1], af[1][2] = af[1][0], af[1][3] = af[1][1];
      } else {
        lds_x4<KSTR>(a1, kstr, af[0][2], af[0][3], af[1][2], af[1][3]);
      }
      uint32_t bq[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if constexpr (DS) {  // (one column block)
          const uint2 f = qfrag[kb * 32 + lane];
          bq[nb][0] = f.x;
          bq[nb][1] = f.y;
        } else {
          bq[nb][0] = qb[kb][nb][0];
          bq[nb][1] = qb[kb][nb][1];
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        af[mt][0] = slot_f16x2(af[mt][0], d0, m0);
        af[mt][1] = slot_f16x2(af[mt][1], d0, m0);
        af[mt][2] = slot_f16x2(af[mt][2], d1, m1);
        af[mt][3] = slot_f16x2(af[mt][3], d1, m1);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) mma_f16(acc[mt][kb & 1][nb], af[mt], bq[nb][0], bq[nb][1]);
      }
    }
    // z/s words of this lane's four tokens (rows gid + 8 m): key records, and the value records' halves
    uint32_t kzw[4], vzw[4];
    lds_x4<KSTR>(sb + kzo, kstr, kzw[0], kzw[1], kzw[2], kzw[3]);
    lds_x4<VSTR>(sb + vzo, vstr, vzw[0], vzw[1], vzw[2], vzw[3]);
    float zk[4], sk[4], zv[4], sv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 fk = __half22float2(*reinterpret_cast<const __half2*>(&kzw[m]));
      const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&vzw[m]));
      zk[m] = fk.x;
      sk[m] = fk.y;
      zv[m] = fv.x;
      sv[m] = fv.y;
    }
    // ---- logits, online softmax, W = p s_V as packed fp16 (hi, lo), this stage's shares of Z and S; FULL: every
    // token of the warp's block is in the split (no masking) ----
    float corr[NB];
    uint32_t pk[4][NB];
    auto softmax = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      bool val[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) val[m] = FULL || r0 + gid + 8 * m < n_in;
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
        float ps = 0.f, pz = 0.f, pw = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float p = ex2_approx(l[nb][m] - m_run[nb]);  // 0 for a masked token
          const float w = val[m] ? p * sv[m] : 0.f;
          ps += p;
          pz += val[m] ? p * zv[m] : 0.f;
          pw += w;
          const __half hi = __float2half_rn(w);
          const __half lo = __float2half_rn(w - __half2float(hi));
          pk[m][nb] = pack_half2(hi, lo);
        }
        l_run[nb] = fmaf(l_run[nb], corr[nb], ps);
        zsum[nb] = fmaf(zsum[nb], corr[nb], pz);
        ssum[nb] = fmaf(ssum[nb], corr[nb], pw);
      }
    };
    if (r0 + WTOK <= n_in)
      softmax(std::true_type{});
    else
      softmax(std::false_type{});
    // ---- W into the value MMA's B layout: k = tile tokens 2 tig, 2 tig + 1 (+8), n = column gid ----
    uint32_t bp[2][NB][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const uint32_t x0 = __shfl_sync(0xffffffffu, pk[2 * mt][nb], srcA);
        const uint32_t x1 = __shfl_sync(0xffffffffu, pk[2 * mt][nb], srcB);
        const uint32_t x2 = __shfl_sync(0xffffffffu, pk[2 * mt + 1][nb], srcA);
        const uint32_t x3 = __shfl_sync(0xffffffffu, pk[2 * mt + 1][nb], srcB);
        bp[mt][nb][0] = __byte_perm(x0, x1, psel);
        bp[mt][nb][1] = __byte_perm(x2, x3, psel);
      }
    // ---- M_j += W A_j: A = value codes (16 channels x 16 tokens) per m-tile; the stage's 32-token products are
    // summed by the MMA from zero and folded into the running sums by round-to-nearest FMAs (acc = acc corr +
    // stage): accumulating inside the MMA across all stages would bias these sums of positive terms by a rounding
    // step per stage, which the near-cancellation of Z, S and M in the output magnifies ----
#pragma unroll
    for (int mb = 0; mb < NBLK; ++mb) {
      if (mb >= nmb) break;  // blocks past the set's last nonzero-width value channel
      // m-tile mt: records 8 mt + tig (tokens 2 tig, +1) and 8 mt + 4 + tig; channels gid (slot 0), gid + 8 (slot 1)
      uint32_t d0, m0, d1, m1, a0, a1;
      if constexpr (DS) {
        const uint4 e = reinterpret_cast<const uint4*>(vtab)[mb * 8 + gid];
        d0 = e.x, m0 = e.y, d1 = e.z, m1 = e.w;
        a0 = sb + vrow + (d0 >> 5), a1 = sb + vrow + (d1 >> 5);
      } else {
        d0 = vd[mb][0], m0 = vm[mb][0], d1 = vd[mb][1], m1 = vm[mb][1];
        a0 = sb + (d0 >> 5), a1 = sb + (d1 >> 5);
      }
      uint32_t af[2][4];
      lds_x4<VSTR>(a0, vstr, af[0][0], af[0][2], af[1][0], af[1][2]);
      if ((SW & 2) || ((smask >> (8 + mb)) & 1u)) {  // both channels in the words just loaded
        af[0][1] = af[0][0], af[0][3] = af[0][2], af[1][1] = af[1][0], af[1][3] = af[1][2];
      } else {
        lds_x4<VSTR>(a1, vstr, af[0][1], af[0][3], af[1][1], af[1][3]);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        af[mt][0] = slot_f16x2(af[mt][0], d0, m0);
        af[mt][1] = slot_f16x2(af[mt][1], d1, m1);
        af[mt][2] = slot_f16x2(af[mt][2], d0, m0);
        af[mt][3] = slot_f16x2(af[mt][3], d1, m1);
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        float tile[4];
        mma_f16_zero(tile, af[0], bp[0][nb][0], bp[0][nb][1]);
        mma_f16(tile, af[1], bp[1][nb][0], bp[1][nb][1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) vacc[mb][nb][e] = fmaf(vacc[mb][nb][e], corr[nb], tile[e]);
      }
    }
    release_stage(i);
  }

  __syncthreads();
  const DecEpi E = decode_epi(NW, NT, !CL);
  float* const fs = reinterpret_cast<float*>(smem);
  float* wpart = fs + E.wpart;  // [NW][g][PSTR]
  float* mrg = fs + E.mrg;      // [g][PSTR]: the CTA's m, l, Z, S, M (rotated basis)
  float* mg = fs + E.mg;        // [8][128]: merged M
  float* hs = fs + E.hs;        // [8][4]: merged l, Z, S
  float* esw = fs + E.esw;      // [MAX_SPLITS][8]: split weights
  float* rot = fs + E.rot;
  float* outp = a.out + ((size_t)b * a.Hq + (size_t)kh * g) * D;  // (b: the virtual sequence)
  if (s_abort) {  // drain the copies this CTA may still have in flight, then leave an empty partial
    if (tid == 0) {
      const int issued = s_issued;
      for (int i = max(0, issued - NS); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % NS]), (uint32_t)((i / NS) & 1), a.wait_ns);
    }
    __syncthreads();
    for (int idx = tid; idx < g * PSTR; idx += NT) mrg[idx] = (idx % PSTR) == 0 ? -INFINITY : 0.f;
  } else {
    // ======== the warps' partials (rotated basis) into shared memory: the ring is consumed ========
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float lsum = l_run[nb], zt = zsum[nb], st = ssum[nb];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        zt += __shfl_xor_sync(0xffffffffu, zt, o);
        st += __shfl_xor_sync(0xffffffffu, st, o);
      }
      const int h = tig + 4 * nb;
      if (h < g) {
        float* w = wpart + (warp * g + h) * PSTR;
        if (gid == 0) {
          w[0] = m_run[nb];
          w[1] = lsum;
          w[2] = zt;
          w[3] = st;
        }
#pragma unroll
        for (int mb = 0; mb < NBLK; ++mb)
          if (mb < nmb) {  // rows gid and gid + 8 of block mb hold the channels vidx[mb][gid][0, 1]
            w[4 + vidx[(mb * 8 + gid) * 2]] = vacc[mb][nb][0] + vacc[mb][nb][1];
            w[4 + vidx[(mb * 8 + gid) * 2 + 1]] = vacc[mb][nb][2] + vacc[mb][nb][3];
          }
      }
    }
    __syncthreads();
    // ---- the CTA's partial: the warps' sums weighted by 2^(m_w - max_w m_w) ----
    const int icols = 4 + nzV;
    for (int idx = tid; idx < g * icols; idx += NT) {
      const int h = idx / icols, cidx = idx - h * icols;
      float mw[NW];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        mw[w] = wpart[(w * g + h) * PSTR];
        M = fmaxf(M, mw[w]);
      }
      float val = M;
      if (cidx > 0) {
        val = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float e = (mw[w] == -INFINITY) ? 0.f : ex2_approx(mw[w] - M);
          val = fmaf(e, wpart[(w * g + h) * PSTR + cidx], val);
        }
      }
      mrg[h * PSTR + cidx] = val;
    }
  }

  if constexpr (CL) {
    // ======== the cluster's splits merge through distributed shared memory; CTA r finishes columns
    // [r 128 / CS, (r + 1) 128 / CS) of every head ========
    cp_async_wait_all();  // this thread's share of the T'_V columns has landed
    cluster_sync_all();   // every split's partial is complete (and every thread's copies, CTA-wide)
    const uint32_t mrg_a = smem_u32(mrg);
    if (warp < g) {  // head h = warp, lane = split: weights e_s = 2^(m_s - max m), merged l, Z, S
      const int h = warp;
      const bool in = lane < CS;
      const uint32_t ra = dsmem_addr(mrg_a + (uint32_t)(h * PSTR) * 4u, in ? lane : 0);
      const float ms = in ? ld_dsmem(ra) : -INFINITY;
      const float ls = in ? ld_dsmem(ra + 4) : 0.f, zs = in ? ld_dsmem(ra + 8) : 0.f, ss = in ? ld_dsmem(ra + 12) : 0.f;
      const float M = warp_max(ms);
      const float e = ms == -INFINITY ? 0.f : ex2_approx(ms - M);
      const float den = warp_sum(e * ls), zt = warp_sum(e * zs), st = warp_sum(e * ss);
      if (in) esw[lane * MAX_G + h] = e;
      if (lane == 0) {
        hs[h * 4 + 0] = den;
        hs[h * 4 + 1] = zt;
        hs[h * 4 + 2] = st;
      }
    }
    for (int idx = tid; idx < MAX_G * D; idx += NT) mg[idx] = 0.f;
    __syncthreads();
    switch (CS) {  // merged M_j
      case 16: cluster_merge_m<16, NT>(mrg_a, esw, mg, g, nzV); break;
      case 8: cluster_merge_m<8, NT>(mrg_a, esw, mg, g, nzV); break;
      case 4: cluster_merge_m<4, NT>(mrg_a, esw, mg, g, nzV); break;
      case 2: cluster_merge_m<2, NT>(mrg_a, esw, mg, g, nzV); break;
      default: cluster_merge_m<1, NT>(mrg_a, esw, mg, g, nzV); break;
    }
    cluster_sync_all();  // no split reads another's partial after this: each may finish and exit
    const int KW = D / CS;
    const float* tsl = reinterpret_cast<const float*>(smem + L.tsl);
    rotate_out<NT>(tsl, tsl + D * KW, mg, hs, rot, g, KW, split * KW, nzV, outp);
  } else {
    // ======== the splits merge through the workspace: each leaves (m, l, Z, S, M) there, the last to arrive
    // merges them and maps the result to the original basis ========
    float* part = a.part + ((size_t)bh * a.splits + split) * g * PSTR;
    for (int idx = tid; idx < g * (4 + nzV); idx += NT) {
      const int h = idx / (4 + nzV), c = idx - h * (4 + nzV);
      part[h * PSTR + c] = mrg[h * PSTR + c];
    }
    // arrival: thread 0's acquire-release add at GPU scope publishes the CTA's partial (ordered before it by the
    // barrier) and, in the last CTA, makes the other splits' partials visible to the whole CTA after the next
    // barrier
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
    // the splits' partials in chunks of up to 32 splits, each staged by one round of 16-byte copies: warp h keeps
    // head h's running maximum M_h, weights e_s = 2^(m_s - M_h) and the running l, Z, S; every thread keeps its
    // items' sums of e_s M_sj
    const float* pb = a.part + (size_t)bh * a.splits * g * PSTR;
    const int S = a.splits;
    float* chunk = fs + E.chunk;
    float* tfull = fs + E.tfull;
    const int per = min(32, (int)(MERGE_CHUNK / (uint32_t)(g * PSTR)));  // splits per chunk
    constexpr int IT = (MAX_G * D + NT - 1) / NT;
    float accI[IT];
#pragma unroll
    for (int r = 0; r < IT; ++r) accI[r] = 0.f;
    float M_run = -INFINITY, den = 0.f, zt = 0.f, st = 0.f;
    for (int idx = tid; idx < MAX_G * D; idx += NT) mg[idx] = 0.f;
    for (int s0 = 0; s0 < S; s0 += per) {
      const int n = min(per, S - s0);
      __syncthreads();  // the previous chunk is consumed
      {
        const uint32_t cdst = smem_u32(chunk);
        const float* src = pb + (size_t)s0 * g * PSTR;
        for (int c = tid; c < n * g * PSTR / 4; c += NT) cp_async16(cdst + 16u * c, src + 4 * c);
        cp_async_commit();
        if (s0 == 0) {  // T'_V and T_V^T mu, w, w2 (all 128 columns) follow the first chunk, landing meanwhile
          const uint32_t tdst = smem_u32(tfull);
          for (int c = tid; c < (D + 3) * (D / 4); c += NT) {
            const int row = c >> 5, cc = c & 31;
            const float* tsrc =
                row < D ? TV.Tsc + (so + row) * D : (row == D ? TV.base : row == D + 1 ? TV.wsum : TV.wsum2) + so;
            cp_async16(tdst + (uint32_t)(row * D + 4 * cc) * 4u, tsrc + 4 * cc);
          }
          cp_async_commit();
          cp_async_wait_prior();
        } else {
          cp_async_wait_all();
        }
      }
      __syncthreads();
      if (warp < g) {
        const int h = warp;
        const float* ph = chunk + (size_t)min(lane, n - 1) * g * PSTR + h * PSTR;
        const float ms = lane < n ? ph[0] : -INFINITY;
        const float Mn = fmaxf(M_run, warp_max(ms));
        const float sc = (M_run == Mn) ? 1.f : exp2f(M_run - Mn);
        const float e = ms == -INFINITY ? 0.f : exp2f(ms - Mn);
        den = fmaf(den, sc, warp_sum(e * ph[1]));
        zt = fmaf(zt, sc, warp_sum(e * ph[2]));
        st = fmaf(st, sc, warp_sum(e * ph[3]));
        M_run = Mn;
        if (lane < n) esw[lane * MAX_G + h] = e;
        if (lane == 0) hs[h * 4 + 3] = sc;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < IT; ++r) {
        const int idx = tid + NT * r;
        if (idx < g * nzV) {
          const int h = idx / nzV, j = idx - h * nzV;
          float acc = accI[r] * hs[h * 4 + 3];
          for (int sp = 0; sp < n; ++sp) acc = fmaf(esw[sp * MAX_G + h], chunk[(sp * g + h) * PSTR + 4 + j], acc);
          accI[r] = acc;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < IT; ++r) {
      const int idx = tid + NT * r;
      if (idx < g * nzV) mg[(idx / nzV) * D + idx % nzV] = accI[r];
    }
    if (warp < g && lane == 0) {
      hs[warp * 4 + 0] = den;
      hs[warp * 4 + 1] = zt;
      hs[warp * 4 + 2] = st;
    }
    cp_async_wait_all();
    __syncthreads();
    rotate_out<NT>(tfull, tfull + D * D, mg, hs, rot, g, D, 0, nzV, outp);
  }
}

#ifndef KVTC_DECODE_KERNELS
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
  split_plan(B, Hkv, T_cap, device, WTOK, 1, MAX_SPLITS, &L.splits, &L.chunk);
  const size_t bh = (size_t)B * Hkv;
  size_t o = 0;
  L.off_cnt = o;
  o = align256(o + bh * sizeof(unsigned));
  L.off_part = o;
  o = align256(o + bh * (size_t)L.splits * g * PSTR * sizeof(float));
  L.total = o;
  return L;
}
#endif

#ifdef KVTC_DECODE_KERNELS
// Largest number of clusters of cs CTAs of kernel fn (with this launch's block and shared memory) that the device
// holds at once; asked once per (kernel, shared memory, cluster size, device). 0 when the device cannot run one.
static int max_active_clusters(const void* fn, const cudaLaunchConfig_t& base, int cs) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, size_t, int, int>, int> known;
  const int dev = current_device();
  const auto key = std::make_tuple(fn, base.dynamicSmemBytes, cs, dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = known.find(key);
    if (it != known.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = base;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    n = 0;
    cudaGetLastError();  // the query's error is not the caller's
  }
  std::lock_guard<std::mutex> lock(mu);
  known[key] = n;
  return n;
}

// Cluster sizes above eight need the kernel's consent, given once per (kernel, device).
static cudaError_t allow_large_clusters(const void* fn) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, bool> done;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  bool& d = done[{fn, dev}];
  if (d) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) d = true;
  return e;
}

// One launch of decode_kernel<NB, RK, RV, NBLK, *>. The splits of each (sequence, KV head) form a thread-block
// cluster when the device holds all B * Hkv clusters at once with a cluster size that keeps at least half the SMs
// busy (sizes 16, 8, 4, 2, 1 tried in turn, each at most SMs / (B * Hkv)); otherwise (few sequence-head pairs)
// the workspace's split plan applies and the splits merge through global memory. plan != nullptr: fill the plan
// (cluster size or 0, splits, stages, warps, channel blocks, shared memory, clusters held for sizes 16 .. 1 or -1
// when not asked, the single-word kernel flag) and launch nothing.
template <int NB, int RK, int RV, int NBLK, int NW, int SW>
cudaError_t launch_decode_kernel(cudaLaunchConfig_t& cfg, const ParamsDev& P, DecArgs a, int ws_splits,
                                        int32_t* plan) {
  const int rk = P.t[0].r_words, rv = P.t[1].r_words;
  const int bh = a.B * a.Hkv, sms = sm_count(current_device());
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (plan)
    for (int i = 0; i < 12; ++i) plan[i] = i >= 6 && i < 11 ? -1 : 0;
  if (plan) plan[11] = SW;
  if (16 * bh >= sms / 2) {
    const void* fn = (const void*)decode_kernel<NB, RK, RV, NBLK, true, NW, SW>;
    if ((e = allow_large_clusters(fn)) != cudaSuccess) return e;
    const int cap = std::max(1, sms / bh);
    for (int cs = 16, slot = 6; cs >= 1; cs >>= 1, ++slot) {
      if (cs > cap) continue;
      cudaLaunchConfig_t c = cfg;
      const int stages = ring_stages_for(rk, rv, NW, cs);
      c.dynamicSmemBytes = decode_smem(rk, rv, stages, NW, cs).total;
      if (c.dynamicSmemBytes > SMEM_LIMIT || ensure_dyn_smem(fn, c.dynamicSmemBytes) != cudaSuccess) {
        cudaGetLastError();  // this size does not fit: try the next
        continue;
      }
      const int held = cs == 1 ? bh : max_active_clusters(fn, c, cs);
      if (plan) plan[slot] = held;
      if (held < bh) continue;
      if (cs * bh < sms / 2) break;  // too few CTAs: the workspace plan does better
      a.splits = cs;
      a.stages = stages;
      if (plan) {
        plan[0] = cs, plan[1] = cs, plan[2] = stages, plan[3] = NW, plan[4] = NBLK;
        plan[5] = (int32_t)c.dynamicSmemBytes;
        return cudaSuccess;
      }
      c.gridDim.x = (unsigned)cs;
      at[1].id = cudaLaunchAttributeClusterDimension;
      at[1].val.clusterDim.x = (unsigned)cs;
      at[1].val.clusterDim.y = 1;
      at[1].val.clusterDim.z = 1;
      c.attrs = at;
      c.numAttrs = 2;
      return cudaLaunchKernelEx(&c, decode_kernel<NB, RK, RV, NBLK, true, NW, SW>, P, a);
    }
  }
  const void* fn = (const void*)decode_kernel<NB, RK, RV, NBLK, false, NW, SW>;
  a.splits = ws_splits;
  a.stages = ring_stages_for(rk, rv, NW, 0);
  cfg.gridDim.x = (unsigned)ws_splits;
  cfg.dynamicSmemBytes = decode_smem(rk, rv, a.stages, NW, 0).total;
  if (plan) {
    plan[0] = 0, plan[1] = ws_splits, plan[2] = a.stages, plan[3] = NW, plan[4] = NBLK;
    plan[5] = (int32_t)cfg.dynamicSmemBytes;
    return cudaSuccess;
  }
  if ((e = ensure_dyn_smem(fn, cfg.dynamicSmemBytes)) != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_kernel<NB, RK, RV, NBLK, false, NW, SW>, P, a);
}
#else
template <int NB, int RK, int RV, int NBLK, int NW, int SW>
cudaError_t launch_decode_kernel(cudaLaunchConfig_t& cfg, const ParamsDev& P, DecArgs a, int ws_splits, int32_t* plan);
#endif

// The compiled variants of decode_kernel's launcher, X(NB, RK, RV, NBLK, NW, SW, part): record lengths with a
// compile-time kernel (equal key and value budgets of 1.25 - 4 bits/element and the joint key/value splits of the
// Llama-shaped layer at 2.75, 2 and 1.33 bits/element) for each single-word mask, and the generic kernel (RK = RV
// = 0, lengths read at run time) of each warp layout. part: the translation unit that compiles the variant.
#define KVTC_DECODE_RW_LIST(X, NB, NBLK, NW, SW, PART)                                                       \
  X(NB, 5, 5, NBLK, NW, SW, PART) X(NB, 6, 4, NBLK, NW, SW, PART) X(NB, 8, 8, NBLK, NW, SW, PART)             \
  X(NB, 11, 11, NBLK, NW, SW, PART) X(NB, 12, 12, NBLK, NW, SW, PART) X(NB, 16, 16, NBLK, NW, SW, PART)       \
  X(NB, 14, 8, NBLK, NW, SW, PART) X(NB, 10, 6, NBLK, NW, SW, PART)
#define KVTC_DECODE_LAYOUT(X, NB, NBLK, NW, P0, P1)                                                          \
  KVTC_DECODE_RW_LIST(X, NB, NBLK, NW, 0, P0) KVTC_DECODE_RW_LIST(X, NB, NBLK, NW, 1, P0)                    \
  KVTC_DECODE_RW_LIST(X, NB, NBLK, NW, 2, P1) KVTC_DECODE_RW_LIST(X, NB, NBLK, NW, 3, P1)                    \
  X(NB, 0, 0, NBLK, NW, 0, P1)
#define KVTC_DECODE_VARIANTS(X)                                                                             \
  KVTC_DECODE_LAYOUT(X, 1, 4, 16, 0, 1) KVTC_DECODE_LAYOUT(X, 1, 8, 16, 2, 3)                                \
  KVTC_DECODE_LAYOUT(X, 2, 4, 8, 4, 5) KVTC_DECODE_LAYOUT(X, 2, 8, 8, 6, 7)                                  \
  X(1, 0, 0, 4, 8, 0, 0) X(1, 0, 0, 8, 8, 0, 2)

#ifndef KVTC_DECODE_KERNELS
// the compile-time kernel of the table's record lengths and single-word mask, else the generic one
template <int NB, int NBLK, int NW>
static cudaError_t launch_decode_rw(cudaLaunchConfig_t& cfg, const ParamsDev& P, const DecArgs& a, int ws_splits,
                                    int32_t* plan) {
  const int rk = P.t[0].r_words, rv = P.t[1].r_words, sw = P.single_word;
#define KVTC_DECODE_PICK(NB_, K, V, NBLK_, NW_, SW_, PART)        \
  if (rk == (K) && rv == (V) && sw == (SW_))                       \
    return launch_decode_kernel<NB, K, V, NBLK, NW, SW_>(cfg, P, a, ws_splits, plan);
  KVTC_DECODE_RW_LIST(KVTC_DECODE_PICK, NB, NBLK, NW, 0, 0)
  KVTC_DECODE_RW_LIST(KVTC_DECODE_PICK, NB, NBLK, NW, 1, 0)
  KVTC_DECODE_RW_LIST(KVTC_DECODE_PICK, NB, NBLK, NW, 2, 0)
  KVTC_DECODE_RW_LIST(KVTC_DECODE_PICK, NB, NBLK, NW, 3, 0)
#undef KVTC_DECODE_PICK
  return launch_decode_kernel<NB, 0, 0, NBLK, NW, 0>(cfg, P, a, ws_splits, plan);
}

kv_status launch_decode(const ParamsDev& P, const CacheView& c, const void* q, int B, int Hq,
                        const int32_t* seq_lens, const int32_t* q_pos, float scale, float* out, void* ws,
                        const DecodeLayout& L, cudaStream_t s, int32_t* plan) {
  DecArgs a;
  uint8_t* w = static_cast<uint8_t*>(ws);  // null when only planning
  a.c = c;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_lens = seq_lens;
  a.q_pos = q_pos;
  a.cnt = reinterpret_cast<unsigned*>(w + L.off_cnt);
  a.part = reinterpret_cast<float*>(w + L.off_part);
  a.out = out;
  a.wait_ns = g_wait_limit_ns;
  a.B = B;
  a.Hkv = c.Hkv;
  a.Hq = Hq;
  a.g = Hq / c.Hkv;
  a.splits = L.splits;
  a.stages = 2;
  a.scale_log2 = scale * 1.4426950408889634f;
  const int nb = a.g <= 4 ? 1 : 2;
  const int rk = P.t[0].r_words, rv = P.t[1].r_words;
  // four channel blocks when every set's nonzero channels fit them, eight otherwise; sixteen warps for one column
  // block when two 512-token stages of these records fit the ring
  const int nblk = std::max(P.t[0].max_nz, P.t[1].max_nz) <= 64 ? 4 : 8;
  const bool w16 = nb == 1 && 2 * dec_stage_tokens(16) * (rk + rv) * 4 <= RING_BUDGET;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.splits, c.Hkv, B);
  cfg.blockDim = dim3(w16 ? 512 : 256);
  cfg.stream = s;
  cudaError_t e;
  if (w16)
    e = nblk == 4 ? launch_decode_rw<1, 4, 16>(cfg, P, a, L.splits, plan)
                  : launch_decode_rw<1, 8, 16>(cfg, P, a, L.splits, plan);
  else if (nb == 1)  // long records: the generic kernel with eight warps
    e = nblk == 4 ? launch_decode_kernel<1, 0, 0, 4, 8, 0>(cfg, P, a, L.splits, plan)
                  : launch_decode_kernel<1, 0, 0, 8, 8, 0>(cfg, P, a, L.splits, plan);
  else
    e = nblk == 4 ? launch_decode_rw<2, 4, 8>(cfg, P, a, L.splits, plan)
                  : launch_decode_rw<2, 8, 8>(cfg, P, a, L.splits, plan);
  if (plan) {
    if (e != cudaSuccess) {
      set_error("decode plan: %s", cudaGetErrorString(e));
      return KV_ERR_CUDA;
    }
    return KV_OK;
  }
  if (e != cudaSuccess) {
    set_error("decode_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return launch_check("decode_kernel");
}

#endif  // KVTC_DECODE_KERNELS

}  // namespace kvtc
