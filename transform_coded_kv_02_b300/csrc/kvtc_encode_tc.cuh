// Encode on the tensor cores: 128-token tiles, rotation y = X T^T by tcgen05 MMAs, thread-per-token quantiser.
// Part of the single CUDA translation unit of the library (included once by kvtc_kernels.cu).
//
// Method: "KV Cache Compression Through the Lens of Transform Coding" (AATC), Key points (a decorrelating
// orthogonal transform per head, then scalar quantisation of each rotated channel at its allocated width);
// "SPHERICAL KV ..." page, third abstract (NOVA-KV: a fixed per-token bit count).
//
// Work unit = (tensor, sequence, KV head, tile of 128 new tokens). A persistent CTA owns a contiguous run of
// units, so the transform of a (tensor, set) is staged once per run:
//   TMA warp   T = T_hi + T_mid + T_lo (three bf16 matrices [128 channels][128 inputs]) and the bf16 token
//              tile X [128 tokens][128 inputs], all by tiled TMA with 128-byte swizzling, X double-buffered;
//   MMA warp   one thread issues 8 K-steps x 3 splits of tcgen05.mma (M = 128 tokens, N = 128 channels,
//              K = 16) into an fp32 accumulator of 128 tensor-memory columns; NACC accumulators rotate;
//   epilogue   NACC groups of four warps; group g takes every NACC-th unit: thread = token row of the
//              accumulator (tcgen05.ld 32x32b), two passes over the channels (min/max, then codes), codes equal
//              to those of every other quantiser of the library, record words assembled in shared memory by
//              atomic ORs, then copied out row by row.
// bf16 inputs are exact in bf16, and the three-way split represents T to about 24 significant bits, so the
// only difference from an fp32 CUDA-core rotation is the order of the fp32 accumulation.
#pragma once
#include <cudaTypedefs.h>

#include "kvtc_tc.cuh"

namespace kvtc {

constexpr int TC_TILE = 128;           // tokens per unit
constexpr int TC_NSPLIT = 3;           // bf16 terms of T
constexpr int TC_NST = 2;              // X stages
constexpr int TC_NACC_MAX = 4;         // tensor-memory accumulators = epilogue groups (4, or 3 for long records)
constexpr uint32_t TC_OP_BYTES = 128u * 128u * 2u;   // one 128 x 128 bf16 operand (two 64-column boxes)
constexpr uint32_t TC_BOX_BYTES = 128u * 128u;       // one 128-row x 128-byte box

struct EncTcArgs {
  const int64_t* dst_pos;  // [B] (every layer alike)
  CacheView c;
  int Z, n_sets;           // Z: virtual sequences (layers x sequences)
  long long t_new;
  int units, tiles_per_head;
  long long wait_ns;
};

struct EncTcSmem {  // byte offsets from the 1024-byte-aligned base of the dynamic shared memory
  uint32_t x, epi, epi_group, par, bits, stage, total;
};

__host__ __device__ inline EncTcSmem enc_tc_smem(int RK, int RV, int nacc) {
  EncTcSmem s;
  s.x = TC_NSPLIT * TC_OP_BYTES;
  s.epi = s.x + TC_NST * TC_OP_BYTES;
  const uint32_t kw = (uint32_t)TC_TILE * (uint32_t)(RK | 1);
  const uint32_t vw = (uint32_t)(TC_TILE / 2 + 1) * (uint32_t)(2 * RV + 1);
  const uint32_t stage_words = kw > vw ? kw : vw;
  // per channel pair (2i, 2i + 1): pmi float4 {mu, mu', 1/sigma, 1/sigma'} (1/sigma NaN at zero width),
  // ptc float4 {2^b, 2^b', 2^b - 1/2, 2^b' - 1/2}, phh float2 {1/2 - 2^(b-21), ...}, pbits uint2 {byte offset of
  // the code word in the record | bit << 16, ...}
  s.par = 0;
  s.bits = D * 8 + D * 8 + D * 4;
  s.stage = s.bits + D * 4;                    // record staging
  s.epi_group = (s.stage + stage_words * 4 + 127) & ~127u;
  s.total = 1024 + s.epi + (uint32_t)nacc * s.epi_group;  // 1024: alignment slack of the base
  return s;
}

// Same verdict for the 128 threads of an epilogue group (named barrier 1 + group).
__device__ __forceinline__ bool group_all(int group, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(1 + group)
      : "memory");
  return r != 0;
}

// Channel parameters of one (tensor, set) for the epilogue, channel j = the calling thread's row: pmi float4 per
// pair {mu, mu', 1/sigma, 1/sigma'} (1/sigma NaN at zero width, which min and max skip), ptc float4 per pair
// {2^b, 2^b', 2^b - 1/2, 2^b' - 1/2}, phh {1/2 - 2^(b-21)}, pbits {byte offset of the code word in the record |
// bit << 16} (keys: pair slot, the odd channel in the high half; values: channel slot of the record's earlier
// token).
__device__ __forceinline__ void tc_stage_channel(const TensorDev& td, int tensor, int set, int j, float* pmi,
                                                 float* ptc, float* phh, uint32_t* pbits) {
  const size_t so = (size_t)set * D;
  const int w = td.widths[so + j];
  const int jp = j >> 1, jo = j & 1;
  pmi[4 * jp + jo] = td.mu[so + j];
  pmi[4 * jp + 2 + jo] = w > 0 ? td.inv_sigma[so + j] : __int_as_float(0x7fc00000);  // NaN: out of min/max
  ptc[4 * jp + jo] = exp2i(w);
  ptc[4 * jp + 2 + jo] = (float)((1 << w) - 1) + 0.5f;
  phh[j] = 0.5f - exp2i(w - 21);
  uint32_t word, bit;
  if (tensor == 0) {
    const uint32_t dsc = td.slots[so + (j >> 1)];
    word = 1u + (dsc & 255u);
    bit = ((dsc >> 8) & 255u) + 16u * (uint32_t)(j & 1);
  } else {
    const uint32_t dsc = td.slots[so + j];
    word = 2u + (dsc & 255u);
    bit = (dsc >> 8) & 255u;
  }
  if (w == 0) bit = 0u;
  pbits[j] = (4u * word) | (bit << 16);
}

// Quantise and pack one token whose rotated coefficients y_j sit in this thread's tensor-memory lane, columns
// [0, 16 nblk) (the columns past nz hold zero-width channels). Whole warps call it (one token per thread).
// Codes are OR-ed into the record at shared address rec_s (shifted by hsh: 16 for the later token of a value
// record); returns the token's z/s word. Tensor memory is left holding y'.
//   pass 1: y'_j = (y_j - mu_j) * (1/sigma_j), two channels at a time; min / max over b_j > 0; y' back to
//           tensor memory; z = fp16(min), s = fp16(max - z).
//   pass 2: the quantiser's code clamp(floor(RN((y' - z) / s) 2^b), 0, 2^b - 1) formed from
//           u = RN((y' - z) * (RN(1/s) 2^b)), which differs from RN((y' - z) / s) 2^b by at most 3 units of
//           2^-24 relative, i.e. by less than 2^(b-21) where it matters (|u| <= 2^b). u is clamped to
//           [1/2, 2^b - 1/2] first, so floor() yields the clamped code and the clamp ends, being half-integers,
//           are never ties. Only a clamped u within 2^(b-21) of an integer can give a different floor: such
//           tokens are redone with the IEEE division, so the codes equal the quantiser's for the given y.
__device__ __forceinline__ uint32_t tc_quantize_pack_row(uint32_t tacc, int nblk, int nz, const float* pmi,
                                                         const float* ptc, const float* phh, const uint32_t* pbits,
                                                         uint32_t rec_s, uint32_t hsh) {
  float m = INFINITY, M = -INFINITY;
  for (int cb = 0; cb < nblk; ++cb) {
    uint32_t v[16];
    tmem_ld_32x32b_x16(tacc + 16u * cb, v);
    tmem_ld_wait();
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
      const float4 mi = reinterpret_cast<const float4*>(pmi)[8 * cb + jp];
      const float2 yp = f2unpack(f2mul(f2sub(f2pack(__uint_as_float(v[2 * jp]), __uint_as_float(v[2 * jp + 1])),
                                             f2pack(mi.x, mi.y)),
                                       f2pack(mi.z, mi.w)));
      m = fminf(m, fminf(yp.x, yp.y));
      M = fmaxf(M, fmaxf(yp.x, yp.y));
      v[2 * jp] = __float_as_uint(yp.x);
      v[2 * jp + 1] = __float_as_uint(yp.y);
    }
    tmem_st_32x32b_x16(tacc + 16u * cb, v);
  }
  tmem_st_wait();
  __half zh = __ushort_as_half(0), sh = __ushort_as_half(0);
  if (nz > 0) {
    zh = half_sat_rn(__fadd_rn(m, 0.f));
    sh = half_sat_rn(__fsub_rn(M, __half2float(zh)));
  }
  const float zf = __half2float(zh), sf = __half2float(sh);
  const bool coded = sf != 0.f;
  const float rs = coded ? __frcp_rn(sf) : 0.f;
  const uint64_t zz = f2pack(zf, zf), rr = f2pack(rs, rs), hv = f2pack(0.5f, 0.5f);
  bool near = false;
  for (int cb = 0; cb < nblk; ++cb) {
    uint32_t v[16];
    tmem_ld_32x32b_x16(tacc + 16u * cb, v);  // y'
    tmem_ld_wait();
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
      const float4 tc = reinterpret_cast<const float4*>(ptc)[8 * cb + jp];
      const float2 hh = reinterpret_cast<const float2*>(phh)[8 * cb + jp];
      const uint2 pb = reinterpret_cast<const uint2*>(pbits)[8 * cb + jp];
      float2 u = f2unpack(f2mul(f2sub(f2pack(__uint_as_float(v[2 * jp]), __uint_as_float(v[2 * jp + 1])), zz),
                                f2mul(rr, f2pack(tc.x, tc.y))));
      u.x = fminf(fmaxf(u.x, 0.5f), tc.z);
      u.y = fminf(fmaxf(u.y, 0.5f), tc.w);
      const float flx = floorf(u.x), fly = floorf(u.y);
      const float2 t = f2unpack(f2sub(f2sub(f2pack(u.x, u.y), f2pack(flx, fly)), hv));
      near |= (fabsf(t.x) > hh.x) | (fabsf(t.y) > hh.y);
      red_or_shared(rec_s + (pb.x & 0xFFFFu), (uint32_t)flx << ((pb.x >> 16) + hsh));
      red_or_shared(rec_s + (pb.y & 0xFFFFu), (uint32_t)fly << ((pb.y >> 16) + hsh));
    }
  }
  near = near && coded;
  if (__any_sync(0xffffffffu, near)) {  // rare: exact quotients for the near-tie tokens of this warp
    for (int cb = 0; cb < nblk; ++cb) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(tacc + 16u * cb, v);
      tmem_ld_wait();
      if (near) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = 16 * cb + jj;
          const float tb = ptc[4 * (j >> 1) + (j & 1)], cm = ptc[4 * (j >> 1) + 2 + (j & 1)];
          const uint32_t pb = pbits[j];
          const float dq = __fsub_rn(__uint_as_float(v[jj]), zf);
          const uint32_t fast = (uint32_t)floorf(fminf(fmaxf(__fmul_rn(dq, __fmul_rn(rs, tb)), 0.5f), cm));
          const uint32_t exact = (uint32_t)floorf(fminf(fmaxf(__fmul_rn(__fdiv_rn(dq, sf), tb), 0.5f), cm));
          if (fast != exact) red_xor_shared(rec_s + (pb & 0xFFFFu), (fast ^ exact) << ((pb >> 16) + hsh));
        }
      }
    }
  }
  return (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
}

template <int NACC>
__global__ void __launch_bounds__((4 * NACC + 2) * 32, 1)
    encode_tc_kernel(ParamsDev P, EncTcArgs a, const __grid_constant__ CUtensorMap mx_k,
                     const __grid_constant__ CUtensorMap mx_v, const __grid_constant__ CUtensorMap mt_k,
                     const __grid_constant__ CUtensorMap mt_v) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t x_full[TC_NST], x_empty[TC_NST], acc_full[NACC], acc_empty[NACC];
  __shared__ __align__(8) uint64_t t_full, t_free, mma_fin;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int RK = P.t[0].r_words, RV = P.t[1].r_words;
  const EncTcSmem L = enc_tc_smem(RK, RV, NACC);
  const int tma_warp = 4 * NACC, mma_warp = 4 * NACC + 1;

  // contiguous run of units of this CTA
  const long long U = a.units;
  const int u0 = (int)(U * blockIdx.x / gridDim.x), u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
  const int per_tensor = a.Z * a.c.Hkv * a.tiles_per_head;
  // unit -> (tensor, bh, tile); the transform key (tensor, set) decides when T is restaged
  auto unit_tensor = [&](int u) { return u / per_tensor; };
  auto unit_bh = [&](int u) { return (u - unit_tensor(u) * per_tensor) / a.tiles_per_head; };
  auto unit_tile = [&](int u) { return (u - unit_tensor(u) * per_tensor) % a.tiles_per_head; };
  auto unit_set = [&](int u) { const int bh = unit_bh(u); return view_set(a.c, bh / a.c.Hkv, bh % a.c.Hkv); };
  auto unit_tkey = [&](int u) { return unit_tensor(u) * a.n_sets + unit_set(u); };

  if (tid == 0) {
    for (int s = 0; s < TC_NST; ++s) {
      mbar_init(smem_u32(&x_full[s]), 1);
      mbar_init(smem_u32(&x_empty[s]), 1);
    }
    for (int g = 0; g < NACC; ++g) {
      mbar_init(smem_u32(&acc_full[g]), 1);
      mbar_init(smem_u32(&acc_empty[g]), 4);  // lane 0 of each warp of the group
    }
    mbar_init(smem_u32(&t_full), 1);
    mbar_init(smem_u32(&t_free), 1);
    mbar_init(smem_u32(&mma_fin), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  static_assert(NACC >= 1 && NACC <= 4, "128 tensor-memory columns per accumulator, 512 in all");
  constexpr uint32_t TMEM_COLS = NACC <= 2 ? 256u : 512u;  // 128 columns per accumulator, a power of two
  if (warp == mma_warp) {
    tmem_alloc(smem_u32(&s_tmem), TMEM_COLS);
    tmem_relinquish();
  }
  // record staging starts zeroed; the epilogue re-zeroes it after every copy-out
  for (uint32_t g = 0; g < NACC; ++g) {
    uint32_t* st = reinterpret_cast<uint32_t*>(gbase + L.epi + g * L.epi_group + L.stage);
    for (uint32_t i = tid; i < (L.epi_group - L.stage) / 4; i += blockDim.x) st[i] = 0u;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == tma_warp) {
    // ================= TMA producer (one thread) =================
    if (lane == 0 && u0 < u1) {
      tma_prefetch_map(&mx_k);
      tma_prefetch_map(&mx_v);
      tma_prefetch_map(&mt_k);
      tma_prefetch_map(&mt_v);
      int tloads = 0, issued = 0;
      for (int u = u0; u < u1 && !s_abort; ++u) {
        const int li = u - u0, s = li % TC_NST;
        const int tensor = unit_tensor(u);
        if (u == u0 || unit_tkey(u) != unit_tkey(u - 1)) {
          if (tloads > 0 && !mbar_wait_bounded(smem_u32(&t_free), (uint32_t)((tloads - 1) & 1), a.wait_ns)) {
            s_abort = 1;
            break;
          }
          const CUtensorMap* mt = tensor == 0 ? &mt_k : &mt_v;
          const uint32_t tb = smem_u32(&t_full);
          mbar_expect_tx(tb, TC_NSPLIT * TC_OP_BYTES);
          for (int p = 0; p < TC_NSPLIT; ++p)
            for (int hf = 0; hf < 2; ++hf)
              tma_load_2d(base + p * TC_OP_BYTES + hf * TC_BOX_BYTES, mt, 64 * hf, (unit_set(u) * TC_NSPLIT + p) * D,
                          tb);
          ++tloads;
        }
        if (li >= TC_NST &&
            !mbar_wait_bounded(smem_u32(&x_empty[s]), (uint32_t)((li / TC_NST - 1) & 1), a.wait_ns)) {
          s_abort = 1;
          break;
        }
        const CUtensorMap* mx = tensor == 0 ? &mx_k : &mx_v;
        const int row0 = (int)((long long)unit_bh(u) * a.t_new + (long long)unit_tile(u) * TC_TILE);
        const uint32_t xb = smem_u32(&x_full[s]);
        mbar_expect_tx(xb, TC_OP_BYTES);
        tma_load_2d(base + L.x + s * TC_OP_BYTES, mx, 0, row0, xb);
        tma_load_2d(base + L.x + s * TC_OP_BYTES + TC_BOX_BYTES, mx, 64, row0, xb);
        ++issued;
      }
      // leave no copy in flight: the last loads of every stage and of T complete before the CTA can exit
      for (int i = (issued > TC_NST ? issued - TC_NST : 0); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&x_full[i % TC_NST]), (uint32_t)((i / TC_NST) & 1), a.wait_ns);
      if (tloads > 0) mbar_wait_bounded(smem_u32(&t_full), (uint32_t)((tloads - 1) & 1), a.wait_ns);
    }
  } else if (warp == mma_warp) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0 && u0 < u1) {
      constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
      int tloads = 0;
      for (int u = u0; u < u1 && !s_abort; ++u) {
        const int li = u - u0, s = li % TC_NST, g = li % NACC;
        if (u == u0 || unit_tkey(u) != unit_tkey(u - 1)) {
          if (!mbar_wait_bounded(smem_u32(&t_full), (uint32_t)(tloads & 1), a.wait_ns)) {
            s_abort = 1;
            break;
          }
          ++tloads;
        }
        if (!mbar_wait_bounded(smem_u32(&x_full[s]), (uint32_t)((li / TC_NST) & 1), a.wait_ns)) {
          s_abort = 1;
          break;
        }
        if (li >= NACC &&
            !mbar_wait_bounded(smem_u32(&acc_empty[g]), (uint32_t)((li / NACC - 1) & 1), a.wait_ns)) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(g * 128);
        const uint32_t xs = base + L.x + s * TC_OP_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t koff = (uint32_t)(kk >> 2) * TC_BOX_BYTES + (uint32_t)(kk & 3) * 32u;
          const uint64_t adesc = smem_desc_k128(xs + koff);
#pragma unroll
          for (int p = 0; p < TC_NSPLIT; ++p)
            tc_mma_bf16(d, adesc, smem_desc_k128(base + p * TC_OP_BYTES + koff), IDESC, (kk | p) ? 1u : 0u);
        }
        tc_commit(smem_u32(&x_empty[s]));
        tc_commit(smem_u32(&acc_full[g]));
        if (u + 1 < u1 && unit_tkey(u + 1) != unit_tkey(u)) tc_commit(smem_u32(&t_free));
      }
      // every MMA issued has completed before tensor memory is released
      tc_commit(smem_u32(&mma_fin));
      mbar_wait_bounded(smem_u32(&mma_fin), 0u, a.wait_ns);
    }
  } else {
    // ================= epilogue groups =================
    const int g = warp >> 2, q = warp & 3;
    const int row = 32 * q + lane;  // accumulator lane = token row of the tile
    uint8_t* eg = gbase + L.epi + g * L.epi_group;
    float* const pmi = reinterpret_cast<float*>(eg + L.par);       // [64][4]
    float* const ptc = pmi + 4 * (D / 2);                            // [64][4]
    float* const phh = ptc + 4 * (D / 2);                            // [64][2]
    uint32_t* const pbits = reinterpret_cast<uint32_t*>(eg + L.bits);  // [64][2]
    uint32_t* stage = reinterpret_cast<uint32_t*>(eg + L.stage);
    int cached_key = -1, k = 0;
    for (int u = u0 + g; u < u1; u += NACC, ++k) {
      const int tensor = unit_tensor(u), bh = unit_bh(u), tile = unit_tile(u), set = unit_set(u);
      const TensorDev& td = P.t[tensor];
      const int R = td.r_words;
      const int z = bh / a.c.Hkv, hk = bh - z * a.c.Hkv;
      if (unit_tkey(u) != cached_key) {  // this group's channel parameters (the group is idle here)
        tc_stage_channel(td, tensor, set, row, pmi, ptc, phh, pbits);
        cached_key = unit_tkey(u);
        named_bar(1 + g, 128);
      }
      const int nz = td.nz[set];
      const int nblk = (nz + 15) >> 4;  // 16-column blocks; channels past nz have width 0
      const bool ok = group_all(g, mbar_wait_bounded(smem_u32(&acc_full[g]), (uint32_t)(k & 1), a.wait_ns));
      if (!ok) {
        s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(g * 128);
      const long long pos0 = a.dst_pos[z % a.c.B] + (long long)tile * TC_TILE;
      const int half = (int)((pos0 + row) & 1);
      const int lr = (row + (int)(pos0 & 1)) >> 1;  // local two-token record of a value token
      const int PK = R | 1, PV = 2 * R + 1;
      uint32_t* const rec = tensor == 0 ? stage + row * PK : stage + lr * PV;
      const uint32_t hsh = tensor == 0 ? 0u : 16u * (uint32_t)half;  // value token: its half of each code word
      const uint32_t zs = tc_quantize_pack_row(tacc, nblk, nz, pmi, ptc, phh, pbits, smem_u32(rec), hsh);
      // the accumulator is free for the next unit of this group
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[g]));
      rec[tensor == 0 ? 0 : half] = zs;
      named_bar(1 + g, 128);
      // ---- copy-out: in a dense cache the tile's records are contiguous and the group copies them word by word;
      // in a paged one record by record, each at its page ----
      const int n_valid = (int)min((long long)TC_TILE, a.t_new - (long long)tile * TC_TILE);
      const int gt = tid & 127;  // thread index within the group
      const long long T_cap = a.c.T_cap;
      const bool dense_run = a.c.bt == nullptr && pos0 >= 0 && pos0 + n_valid <= T_cap;
      if (tensor == 0) {
        uint32_t* dst = a.c.rec[0] + (size_t)bh * (a.c.bt ? 0 : T_cap) * R;  // (dense)
        if (dense_run) {
          const uint32_t mR = 0xFFFFFFFFu / (uint32_t)R + 1u;  // i / R = umulhi(i, mR) for i < 2^16
          uint32_t* d0 = dst + pos0 * R;
          for (int i = gt; i < n_valid * R; i += 128) {
            const int r = (int)__umulhi((uint32_t)i, mR);
            d0[i] = stage[r * PK + (i - r * R)];
          }
        } else {
          for (int r = gt; r < n_valid; r += 128) {
            const long long pos = pos0 + r;
            uint32_t* out = pos >= 0 && pos < T_cap ? view_key_record(a.c, z, hk, pos, R) : nullptr;
            if (!out) {
              atomicOr(&g_status, ST_BAD_INDEX);
              continue;
            }
            for (int w = 0; w < R; ++w) out[w] = stage[r * PK + w];
          }
        }
      } else {
        // local record r holds tokens 2r - odd and 2r - odd + 1 of the tile; the first and the last record may
        // hold only one of this tile's tokens (their other halves belong to neighbouring writes)
        uint32_t* dst = a.c.rec[1] + (size_t)bh * (a.c.bt ? 0 : T_cap / 2) * 2 * R;  // (dense)
        const int odd = (int)(pos0 & 1);
        const int nrec = ((n_valid - 1 + odd) >> 1) + 1;
        const int f0 = odd, f1 = ((n_valid + odd) & 1) ? nrec - 1 : nrec;  // full records [f0, f1)
        const long long gr0 = pos0 >> 1;  // global record of local record 0 (rounds toward minus infinity)
        if (dense_run) {
          const int W2 = 2 * R;
          const uint32_t mW = 0xFFFFFFFFu / (uint32_t)W2 + 1u;
          uint32_t* d0 = dst + (gr0 + f0) * W2;
          for (int i = gt; i < (f1 - f0) * W2; i += 128) {
            const int r = (int)__umulhi((uint32_t)i, mW);
            d0[i] = stage[(f0 + r) * PV + (i - r * W2)];
          }
          // partial records (never the same one): the first holds only its later token when pos0 is odd, the
          // last only its earlier token when the tile ends on an even position; copy this tile's half of each
          // code word and its z/s word
          for (int e = 0; e < 2; ++e) {
            if (e == 0 ? odd == 0 : f1 != nrec - 1) continue;
            const int r = e == 0 ? 0 : nrec - 1, hh = e == 0 ? 1 : 0;
            const uint32_t* src = stage + r * PV;
            uint32_t* drec = dst + (gr0 + r) * W2;
            for (int w = gt; w < W2; w += 128) {
              if (w < 2) {
                if (w == hh) drec[w] = src[w];
              } else {
                reinterpret_cast<uint16_t*>(drec)[2 * w + hh] = reinterpret_cast<const uint16_t*>(src)[2 * w + hh];
              }
            }
          }
        } else {
          for (int r = gt; r < nrec; r += 128) {
            for (int hh = 0; hh < 2; ++hh) {
              const int tr = 2 * r - odd + hh;
              if (tr < 0 || tr >= n_valid) continue;
              const long long pos = pos0 + tr;
              uint32_t* drec = pos >= 0 && pos < T_cap ? view_value_record(a.c, z, hk, pos, R) : nullptr;
              if (!drec) {
                atomicOr(&g_status, ST_BAD_INDEX);
                continue;
              }
              const uint32_t* src = stage + r * PV;
              drec[hh] = src[hh];
              for (int w = 2; w < 2 * R; ++w)
                reinterpret_cast<uint16_t*>(drec)[2 * w + hh] = reinterpret_cast<const uint16_t*>(src)[2 * w + hh];
            }
          }
        }
      }
      named_bar(1 + g, 128);
      // zero the staging words this unit used, for the next one
      {
        const int words = tensor == 0 ? TC_TILE * PK : (TC_TILE / 2 + 1) * PV;
        for (int i = row; i < words; i += 128) stage[i] = 0u;
      }
      named_bar(1 + g, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == mma_warp) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side: tensor maps and launch ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 matrix [rows][128] (256-byte rows), boxes of box_rows (at most 128 and at most rows) x 64 columns,
// 128-byte swizzle, zero fill past the last row
static bool make_bf16_map(CUtensorMap* m, const void* ptr, unsigned long long rows, unsigned box_rows = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NACC>
static cudaError_t launch_encode_tc_n(const ParamsDev& P, const EncTcArgs& a, const CUtensorMap* maps,
                                      uint32_t smem, cudaStream_t s, int grid) {
  cudaError_t e = ensure_dyn_smem((const void*)encode_tc_kernel<NACC>, smem);
  if (e != cudaSuccess) return e;
  encode_tc_kernel<NACC><<<grid, (4 * NACC + 2) * 32, smem, s>>>(P, a, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

// Tensor-core encode of bf16 tokens. Returns KV_ERR_UNSUPPORTED (nothing launched) when the shapes fall outside
// what the kernel handles, so the caller can take the CUDA-core path.
static kv_status launch_encode_tc(const ParamsDev& P, const CacheView& c, const void* k, const void* v, int Z,
                                  int64_t t_new, const int64_t* dst_pos, cudaStream_t s) {
  const long long rows = (long long)Z * c.Hkv * t_new;
  if (rows + TC_TILE >= (1LL << 31) || P.n_sets * TC_NSPLIT * D >= (1 << 30)) {
    set_error("tensor-core encode: %lld token rows exceed the kernel's 32-bit tile coordinates", rows);
    return KV_ERR_UNSUPPORTED;
  }
  const int RK = P.t[0].r_words, RV = P.t[1].r_words;
  // four epilogue groups (18 warps, 96 registers a thread) where their record staging fits in shared memory,
  // else three (14 warps), which fit for every record length up to 33 words
  const int nacc = enc_tc_smem(RK, RV, TC_NACC_MAX).total <= 227u * 1024u ? TC_NACC_MAX : TC_NACC_MAX - 1;
  const uint32_t smem = enc_tc_smem(RK, RV, nacc).total;
  if (smem > 227u * 1024u) {
    set_error("tensor-core encode: %u bytes of shared memory needed", smem);
    return KV_ERR_UNSUPPORTED;
  }
  CUtensorMap maps[4];
  if (!make_bf16_map(&maps[0], k, (unsigned long long)rows) || !make_bf16_map(&maps[1], v, (unsigned long long)rows) ||
      !make_bf16_map(&maps[2], P.t[0].Tsplit, (unsigned long long)P.n_sets * TC_NSPLIT * D) ||
      !make_bf16_map(&maps[3], P.t[1].Tsplit, (unsigned long long)P.n_sets * TC_NSPLIT * D)) {
    set_error("tensor-core encode: tensor map encoding failed");
    return KV_ERR_UNSUPPORTED;
  }
  EncTcArgs a;
  a.dst_pos = dst_pos;
  a.c = c;
  a.Z = Z;
  a.n_sets = P.n_sets;
  a.t_new = t_new;
  a.tiles_per_head = (int)((t_new + TC_TILE - 1) / TC_TILE);
  const long long units = 2LL * Z * c.Hkv * a.tiles_per_head;
  if (units >= (1LL << 31)) {
    set_error("tensor-core encode: too many tiles");
    return KV_ERR_UNSUPPORTED;
  }
  a.units = (int)units;
  a.wait_ns = g_wait_limit_ns;
  const int grid = (int)std::min<long long>(units, sm_count(current_device()));
  const cudaError_t e = nacc == TC_NACC_MAX ? launch_encode_tc_n<TC_NACC_MAX>(P, a, maps, smem, s, grid)
                                            : launch_encode_tc_n<TC_NACC_MAX - 1>(P, a, maps, smem, s, grid);
  if (e != cudaSuccess) {
    set_error("encode_tc_kernel launch: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

}  // namespace kvtc
