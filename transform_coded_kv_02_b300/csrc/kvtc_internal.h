// Internal declarations shared by the host library (kvtc_host.cpp) and the kernels (kvtc_kernels.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/kvtc.h"

namespace kvtc {

constexpr int D = 128;          // head dimension
constexpr int MAX_BITS = 8;     // largest channel width in the library
constexpr int MAX_G = 8;        // query heads per KV head
constexpr int MAX_RW = 1 + MAX_BITS * D / 32;  // 33 record words

// device status bits (read by kv_check_status)
constexpr unsigned ST_TIMEOUT = 1u;
constexpr unsigned ST_BAD_INDEX = 2u;

// One tensor's (K or V) parameters for all sets, device pointers. Arrays are set-major.
struct TensorDev {
  const float* T;                  // [S][D][D]  rows = storage channels
  const float* TT;                 // [S][D][D]  TT[k][j] = T[j][k]
  const float* Tq;                 // [S][D][D]  Tq[k][j] = (T^-1)[k][j]: the decode's q~ = T^-T q (TT when T is
                                   //            orthogonal)
  const __nv_bfloat16* Tsplit;     // [S][3][D][D]  T = hi + mid + lo, each bf16
  const float* mu;                 // [S][D]  rotated means (storage order)
  const float* sigma;              // [S][D]
  const float* inv_sigma;          // [S][D]  fp32(1/sigma) computed in double; 0 for zero-width
  const float* base;               // [S][D]  T^-1 mu (original-basis vector of the all-mean record)
  const float* Tsc;                // [S][D][D]  (T^-1)[k][j] sigma_j at [j][k] (0 for zero-width rows)
  const float* wsum;               // [S][D]  sum over b_j > 0 of (T^-1)[k][j] sigma_j
  const float* wsum2;              // [S][D]  sum over b_j > 0 of (T^-1)[k][j] sigma_j (2^(w_j - b_j) - 2^(-b_j - 1)),
                                   //         w_j = slot width (keys: the pair's wider width; values: b_j)
  const float* smax;               // [S]     max over b_j > 0 of sigma_j 2^(w_j - b_j)
  const uint8_t* widths;           // [S][D]
  const int32_t* nz;               // [S]     1 + last storage channel with width > 0
  const uint32_t* slots;           // [S][D] slots: code word | bit << 8 | b_lo << 16 | b_hi << 24; keys: entry k =
                                   // channel pair (2k, 2k+1) of a one-token record (k < D/2); values: entry j =
                                   // channel j of a two-token record (code words start at record word 2)
  const uint32_t* slp;             // [S][8 blocks][lanes][2] slot descriptors in the decode's lane order (keys:
                                   //   4 lanes of pair slots, values: 8 lanes of channels)
  const uint8_t* idx;              // [S][8][lanes][2] the pair (keys) or channel (values) at each position
  const uint32_t* single;          // [S] blocks whose lane couples share a code word: keys bits 0-7, values 8-15
                                   //   (the same array in both tensors)
  int r_words;                     // record words per token (same for every set)
  int min_nz;                      // smallest nz over the sets
  int max_nz;                      // largest nz over the sets
};

struct ParamsDev {
  TensorDev t[2];
  int n_sets;
  // rotary embedding of the decode's queries: frequency i (pairs (i, i + D/2)) as a fraction of a turn in 64-bit
  // fixed point, turns_i = round(base^(-2i/D) / (2 pi) 2^64) [D/2]; null when the table has no embedding
  const unsigned long long* rope_turns;
  // bit 0: in every set, every key channel block the decode reads takes both slots of each lane from one code word
  // (TensorDev::single); bit 1: the same for the value blocks
  int single_word;
};

// Where a launch's records live and which parameter set serves them, built by the entry points from a kv_cache
// (dense) or a kv_paged_cache. A launch covers Z virtual sequences z = l * B + b (layer l of the view, sequence b).
struct CacheView {
  uint32_t* rec[2];      // dense: [Z][Hkv][T_cap] records (values: two-token records); paged: the page pools
  const int32_t* bt;     // paged: block table [Z][max_pages]; null: dense
  long long T_cap;       // positions per (z, KV head): the dense capacity, or max_pages * P
  long long n_pages;     // pages in each pool (paged)
  int P;                 // tokens per page (paged: a power of two, at least 32)
  int P_shift;           // log2 P
  int max_pages;
  int B;                 // sequences per layer: z % B indexes write positions, lengths and query positions
  int Hkv;
  int per_seq;           // one parameter set per (sequence, KV head) instead of per KV head
  int set_base;          // parameter set of the view's first layer, KV head 0
  int sets_per_layer;
};
__host__ __device__ inline int view_set(const CacheView& c, int z, int h) {
  const int l = z / c.B, b = z - l * c.B;
  return c.set_base + l * c.sets_per_layer + (c.per_seq ? b * c.Hkv + h : h);
}
// The key record of (z, KV head h, position pos < T_cap), or null when its page index is out of range.
__host__ __device__ inline uint32_t* view_key_record(const CacheView& c, int z, int h, long long pos, int R) {
  if (!c.bt) return c.rec[0] + (((size_t)z * c.Hkv + h) * (size_t)c.T_cap + (size_t)pos) * R;
  const long long pg = c.bt[(size_t)z * c.max_pages + (size_t)(pos >> c.P_shift)];
  if (pg < 0 || pg >= c.n_pages) return nullptr;
  return c.rec[0] + ((((size_t)pg * c.Hkv + h) << c.P_shift) + (size_t)(pos & (c.P - 1))) * R;
}
// The two-token value record holding position pos (R: words per token), or null (page index out of range).
__host__ __device__ inline uint32_t* view_value_record(const CacheView& c, int z, int h, long long pos, int R) {
  if (!c.bt) return c.rec[1] + (((size_t)z * c.Hkv + h) * (size_t)(c.T_cap / 2) + (size_t)(pos >> 1)) * 2 * R;
  const long long pg = c.bt[(size_t)z * c.max_pages + (size_t)(pos >> c.P_shift)];
  if (pg < 0 || pg >= c.n_pages) return nullptr;
  return c.rec[1] + ((((size_t)pg * c.Hkv + h) << (c.P_shift - 1)) + (size_t)((pos & (c.P - 1)) >> 1)) * 2 * R;
}

// First-fit placement of the pair slots of widths w[d] in a record of rw words (word/pos [d/2], -1 = empty);
// false when a slot finds no room.
bool slot_layout(const int32_t* w, int d, int rw, int* word, int* pos);
// First-fit placement of single channels in a two-token value record (word/pos [d]).
bool token_slot_layout(const int32_t* w, int d, int rw, int* word, int* pos);

// host-side error message of the calling thread
void set_error(const char* fmt, ...);
void clear_error();

// Kernel launchers (kvtc_kernels.cu). They assume validated arguments.
// (Z: virtual sequences of the view; k, v: [Z][Hkv][t_new][D])
kv_status launch_encode(const ParamsDev& P, const CacheView& c, const void* k, const void* v, int dtype,
                        int Z, int64_t t_new, const int64_t* dst_pos, int path, cudaStream_t s);
struct DecodeLayout {
  int splits;
  int chunk;                  // tokens per split at full capacity, multiple of the decode tile
  size_t off_cnt, off_part, total;
};
DecodeLayout decode_layout(int B, int Hkv, int Hq, int64_t T_cap, int device);
DecodeLayout decode_bf16_layout(int B, int Hkv, int64_t T_cap, int device);
// (Z: virtual sequences of the view; q, out: [Z][Hq][D]; q_pos: [B] query positions for the rotary embedding, or
// null.) plan != nullptr: fill plan[12] (see kv_debug_decode_plan) and launch nothing
kv_status launch_decode(const ParamsDev& P, const CacheView& c, const void* q, int Z, int Hq,
                        const int32_t* seq_lens, const int32_t* q_pos, float scale, float* out, void* ws,
                        const DecodeLayout& L, cudaStream_t s, int32_t* plan = nullptr);
// the dense view of a kv_cache (one layer, sets per head or per (sequence, head))
CacheView dense_view(const kv_cache& c);
// (dev: receives the current device, which holds the parameter table)
kv_status check_decode_args(const kv_params* p, const kv_cache* c, const void* q, int B, int Hq,
                            const int32_t* seq_lens_dev, float softmax_scale, const float* out, int* dev);
// token-axis allocation: weights workspace (per-run softmax statistics of the observation queries)
struct TokenLayout {
  int nt;  // 128-token tiles per (sequence, KV head)
  size_t off_stats, total;
};
TokenLayout token_layout(int B, int Hkv, int64_t T);
kv_status launch_token_weights(const void* q_obs, int W, const void* k, int B, int Hkv, int Hq, int64_t T,
                               float scale, float* lam, void* ws, cudaStream_t s);
kv_status launch_token_select(const float* lam, int B, int Hkv, int64_t T, int64_t keep, int32_t* idx,
                              cudaStream_t s);
kv_status launch_compact(const ParamsDev& P, const kv_cache& src, const kv_cache& dst, int B, const int32_t* idx,
                         int64_t keep, cudaStream_t s);
kv_status launch_decode_bf16(const void* k, const void* v, int B, int Hkv, int Hq, int64_t T_cap,
                             const void* q, const int32_t* seq_lens, float scale, float* out, void* ws,
                             const DecodeLayout& L, cudaStream_t s);
kv_status launch_debug_quantize_pack(const ParamsDev& P, int set, int tensor, const float* y, int64_t n,
                                     uint32_t* rec, int variant, cudaStream_t s);
kv_status launch_debug_unpack(const ParamsDev& P, int set, int tensor, const uint32_t* rec, int64_t n,
                              uint16_t* codes, cudaStream_t s);
kv_status launch_wait_selftest(cudaStream_t s);
void set_wait_limit_ns(long long ns);
kv_status read_and_clear_device_status(unsigned* out);

// The decode kernel's variants are compiled in DECODE_PARTS translation units (kvtc_decode_part.cu, once per part
// number), each with its own device status word; this reads and clears the one of a part.
constexpr int DECODE_PARTS = 8;
kv_status read_and_clear_decode_status(int part, unsigned* out);

}  // namespace kvtc

// Host-side parameter table.
struct kv_params {
  int d = 0;
  int n_sets = 0;
  int max_bits = 8;
  int r_words[2] = {0, 0};
  std::vector<float> T[2];         // [S][D][D]
  std::vector<float> mu[2];        // [S][D]
  std::vector<float> sigma[2];     // [S][D]
  std::vector<int32_t> widths[2];  // [S][D]
  std::vector<double> eig[2];      // [S][D] variances of the rotated channels (storage order)
  std::vector<double> imp[2];      // [S][D] importances (storage order)
  std::vector<float> Tinv[2];      // [S][D][D] inverse of a non-orthogonal T (Tinv[k][j]: column j pairs with
                                   // storage channel j); empty: T is orthogonal and its inverse is T^T
  double rope_base = 0.0;          // rotary embedding of the decode's queries (0: none)
  int device = -1;
  void* dev_blob = nullptr;
  size_t dev_bytes = 0;
  kvtc::ParamsDev dev{};
};
