/*
 * kvtc.h - C ABI of the transform-coded KV cache library (B300 / sm_103a).
 *
 * Attention-aware transform coding of the KV cache: per (layer, KV head) an orthogonal d x d transform
 * (a KLT of calibration statistics) rotates each token's key and value; each rotated channel is scalar
 * quantised at a width of 0-8 bits chosen by reverse water-filling over attention-aware importances; the
 * codes are bit-packed into fixed-width per-token records; decode attention runs directly over the
 * records.
 *
 * Sources (web pages on the method; they describe it in words only):
 *   [AATC]    "KV Cache Compression Through the Lens of Transform Coding" - At a glance, Key points
 *             (white-noise additive key/value distortion; transform coding + reverse water-filling over a
 *             calibration set), Full text.
 *   [SPECTRA] "SPECTRA: Pushing the KV Cache Beyond the 2-Bit Cliff via Spectral Transform Coding" -
 *             abstract (rotate into a basis computed from the cache's own statistics; concentrate bits).
 *   [RDKV]    "SPHERICAL KV: Angle-Domain Attention and Rate-Distortion Retention ..." - first abstract
 *             (bit widths from full precision down to zero by reverse water-filling, applied once).
 *   [NOVA-KV] same page, third abstract (decode is bandwidth-bound; fixed per-token bit count; transforms
 *             from calibration statistics).
 *
 * Conventions
 *   - d = 128 (head dimension) is the only supported value; g = Hq / Hkv query heads share a KV head
 *     (query head hq reads KV head hq / g); g <= 8.
 *   - Device pointers are owned by the caller. kv_encode and kv_attend_decode never allocate device
 *     memory and never synchronise the host; they enqueue work on the given stream.
 *   - Argument errors are returned synchronously before any launch. Errors raised inside a kernel
 *     (a bounded wait that ran out, a record index out of range) set a per-device status word that
 *     kv_check_status reports (and clears).
 *   - kv_stream_t is a cudaStream_t passed as an opaque pointer (NULL = legacy default stream).
 *   - Every function returns KV_OK (0) on success; kv_last_error() gives a message for the calling
 *     thread's last failure.
 */
#ifndef KVTC_H
#define KVTC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kv_status;
enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer, set index out of range      */
  KV_ERR_UNSUPPORTED = 2, /* d != 128, g > 8, unknown dtype                                           */
  KV_ERR_BUDGET = 3,      /* bits per element gives fewer than 1 or more than 1 + 8*d/32 record words */
  KV_ERR_NUMERIC = 4,     /* non-finite calibration data or statistics                                */
  KV_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed                              */
  KV_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out (reported by kv_check_status)         */
  KV_ERR_IO = 7,          /* parameter file missing, truncated, wrong version or bad checksum         */
  KV_ERR_DEVICE = 8       /* a kernel reported a bad index (reported by kv_check_status)              */
};

enum { KV_DTYPE_F32 = 0, KV_DTYPE_BF16 = 1 };
enum { KV_TENSOR_K = 0, KV_TENSOR_V = 1 };

typedef void* kv_stream_t;

/* ------------------------------------------------------------------------------------------------------
 * Calibration (host).  [AATC Key points 2nd bullet; RDKV; SPECTRA; NOVA-KV]
 * ------------------------------------------------------------------------------------------------------ */

/* Opaque parameter table: for each calibration set and each tensor (K, V) the transform T (rows = storage
 * channels), rotated means mu, standard deviations sigma, channel widths, record length. Owned by the
 * library; free with kv_params_free. */
typedef struct kv_params kv_params;

/* One calibration set (one KV head of one layer, or of one sequence). Host fp32, row-major.
 *   k, v: [n_tok][d] keys and values; q: [n_q][d] query vectors of the g query heads that read this KV
 *   head, stacked (pooled into one second moment). */
typedef struct {
  const float* k;
  const float* v;
  const float* q;
  int64_t n_tok;
  int64_t n_q;
} kv_calib_set;

typedef struct {
  int d;          /* head dimension, must be 128                                                    */
  float bits_k;   /* budget in bits per key element, counting the per-token fp16 scale/zero (2.75 -> 11 words) */
  float bits_v;   /* same for values                                                                */
  int max_bits;   /* largest channel width, 1..8 (8)                                                 */
  int n_threads;  /* host threads for calibration; 0 = all hardware threads                         */
  int joint;      /* 0: keys and values each get their own budget (R_wK from bits_k, R_wV from bits_v).
                   * 1: the table keeps R_wK + R_wV words per token but splits them between keys and values
                   *    jointly (see kv_calibrate)                                                      */
  int key_basis;  /* 0: the KLT of Sigma_K. 1: the attention-aware orthogonal key basis. 2: the non-orthogonal
                   *    key transform (see kv_calibrate) */
} kv_calib_opts;

/* Calibrate n_sets sets: fp64 mean/covariance of K and V, query second moment M_Q, Jacobi
 * eigendecomposition (eigenvalues descending, largest-|.| component of each eigenvector positive),
 * importances lambda_K = sigma^2 * (u^T M_Q u), lambda_V = sigma^2, reverse water-filling to
 * C = 32*R_w - 32 code bits with R_w = floor(bits*d/32), storage order (width desc, lambda desc, index asc).
 * joint = 1 (one rate trade-off between keys and values, [AATC] Key points, first bullet: the attention-aware
 * distortion is a sum of a key and a value part): to first order the output error is
 * sum_t p_t^2 (alpha^2 |v_t - o|^2 sum_i w_i D^K_i + sum_i D^V_i), so with |v_t - o|^2 taken at tr(Sigma_V) and
 * alpha = 1/sqrt(d) the key importances weigh rho = tr(Sigma_V)/d against the value importances. The split
 * R_wK of the table's R_wK + R_wV record words minimises sum over sets of rho sum_i lambda_K,i 4^-b_i +
 * sum_j lambda_V,j 4^-b_j (each tensor water-filled at its own budget); objectives within a relative 1e-9 tie,
 * ties go to the split nearest the separate one, then to fewer key words. The record lengths then differ
 * between keys and values (kv_params_record_words).
 * key_basis = 1 ([NOVA-KV]: derive the key transform from the attention-aware distortion, here kept
 * orthogonal): with white noise in basis U the key distortion is sum_i w_i D_i, and water-filling against the
 * coefficient variances s_i = u_i^T Sigma_K u_i makes it proportional to (prod_i s_i w_i)^(1/d) at high rate.
 * Starting from the KLT, 8 cyclic Jacobi sweeps rotate each pair (i < j) by the angle on a 48-point grid over
 * [-pi/4, pi/4) that minimises the pair's log s_i + log s_j + log w_i + log w_j (rotating only when that gains
 * more than 1e-10); the key importances are then s_i w_i and the stored variances s_i.
 * key_basis = 2 ([NOVA-KV], third abstract: the optimal key transform is not orthogonal and satisfies a
 * generalised Parseval relation): T = c V^T M_Q^(1/2) with V the eigenvectors of M_Q^(1/2) Sigma_K M_Q^(1/2)
 * (M_Q + 1e-12 tr/d I), so that e^T M_Q e = |T e|^2 / c^2 and the coefficients are uncorrelated with
 * variances c^2 lambda; the key importances are those variances. c is the largest column norm of
 * M_Q^(-1/2) V, so every column of T^-1 has norm <= 1. The table keeps T^-1 beside T (kv_params_set_inverse);
 * the encode applies T, the decode rotates q by T^-T.
 * The result lives on the host; call kv_params_upload before encoding or decoding.
 * Errors: KV_ERR_INVALID_ARG (null, n_tok < 2, n_q < 1), KV_ERR_UNSUPPORTED (d), KV_ERR_BUDGET,
 * KV_ERR_NUMERIC (non-finite input). */
kv_status kv_calibrate(int n_sets, const kv_calib_set* sets, const kv_calib_opts* opts, kv_params** out);

/* Build a parameter table from explicit arrays (host, fp32, set-major): T_* [n_sets][d][d] (rows =
 * storage channels), mu_* / sigma_* [n_sets][d], widths_* [n_sets][d] (0..8; the key widths must fit the
 * key record's first-fit pair slots, the value widths the value record's first-fit channel slots, else
 * KV_ERR_BUDGET).
 * Channels with sigma == 0 get width 0. Used to feed externally computed parameters (e.g. by a reference
 * implementation) to the codec. */
kv_status kv_params_from_arrays(int d, int n_sets,
                                const float* T_k, const float* mu_k, const float* sigma_k,
                                const int32_t* widths_k, int r_words_k,
                                const float* T_v, const float* mu_v, const float* sigma_v,
                                const int32_t* widths_v, int r_words_v, kv_params** out);

/* Give tensor (0 = keys, 1 = values) of the table a non-orthogonal transform's inverse: Tinv [n_sets][d][d]
 * host fp32, Tinv[k][j] = (T^-1)[k][j], column j pairing with storage channel j (the same order as T's rows).
 * The decode then uses k^ = T^-1 y^ ([NOVA-KV] non-orthogonal key transform): q is rotated by T^-T, and the
 * folded vectors (T^-1 mu, the column sums of T^-1 sigma) are formed with T^-1. Tinv = NULL removes it (T is then
 * taken as orthogonal, its inverse T^T). Takes effect at the next kv_params_upload; saved by kv_params_save.
 * Errors: KV_ERR_INVALID_ARG (null table, bad tensor, non-finite entries). */
kv_status kv_params_set_inverse(kv_params* p, int tensor, const float* Tinv);
/* Copy one set's inverse of tensor's transform to Tinv [d][d] (host, layout as above). KV_ERR_UNSUPPORTED when the
 * table holds none (an orthogonal transform); KV_ERR_INVALID_ARG for a bad argument. */
kv_status kv_params_get_inverse(const kv_params* p, int set, int tensor, float* Tinv);

/* Rotary position embedding of the decode's queries, for kv_attend_decode_paged with q positions: pairs of
 * channels (i, i + d/2) of q are rotated by the angle pos * base^(-2i/d), i < d/2 (the half-split convention,
 * without frequency rescaling). base > 0 sets it, base = 0 removes it. Takes effect at the next kv_params_upload,
 * which stores the 64 frequencies as fractions of a turn in 64-bit fixed point, so that the angle of any position
 * is reduced exactly before its sine and cosine are taken; saved by kv_params_save. [SPECTRA abstract: longer
 * contexts and larger batches; the in-kernel embedding spares a separate pass over q.] Errors:
 * KV_ERR_INVALID_ARG (null table, negative or non-finite base). */
kv_status kv_params_set_rope(kv_params* p, double base);
double kv_params_get_rope(const kv_params* p);

/* Copy the table to the current CUDA device (allocates device memory owned by the table; the stream
 * orders the copies). Must be called again after switching devices. */
kv_status kv_params_upload(kv_params* p, kv_stream_t stream);

int kv_params_num_sets(const kv_params* p);
int kv_params_record_words(const kv_params* p, int tensor);

/* Read back one set/tensor (host arrays, any may be NULL): widths [d], eigenvalues (variances of the
 * rotated channels, storage order) [d], importances [d], T [d][d], mu [d], sigma [d]. */
kv_status kv_params_info(const kv_params* p, int set, int tensor, int32_t* widths, double* eigvals,
                         double* importance, float* T, float* mu, float* sigma);

/* Versioned binary file with a CRC32 of the payload. */
kv_status kv_params_save(const kv_params* p, const char* path);
kv_status kv_params_load(const char* path, kv_params** out);
void kv_params_free(kv_params* p);

/* ------------------------------------------------------------------------------------------------------
 * Packed cache (device, caller-owned).  [NOVA-KV: fixed per-token bit count and fixed-width layout]
 * z/s word of a token = fp16 zero point z (bits 0-15) | fp16 scale s (bits 16-31); unused bits are 0.
 * Key record (one token, r_words_k words): word 0 = z/s; storage channels (2k, 2k+1) share slot k at bit r_k
 *   of code word 1 + u_k: channel 2k in the low half, channel 2k+1 in the high half.
 * Value record (tokens 2p and 2p+1, 2 r_words_v words): words 0 and 1 = their z/s words; channel j has slot j
 *   at bit r_j of code word 2 + u_j: token 2p's code in the low half, token 2p+1's in the high half. (Decode
 *   contracts values over tokens; this puts the two codes one tensor-core operand register needs into one
 *   word.) Slots are placed first-fit by kv_calibrate / kv_params_from_arrays.
 * ------------------------------------------------------------------------------------------------------ */
typedef struct {
  uint32_t* k_rec;      /* [B][Hkv][T_cap][r_words_k], 16-byte aligned                                 */
  uint32_t* v_rec;      /* [B][Hkv][T_cap / 2][2 r_words_v] (same bytes as T_cap one-token records),
                           16-byte aligned                                                              */
  int B;
  int Hkv;
  int64_t T_cap;        /* token capacity per (sequence, head); multiple of 16                          */
  int per_seq_params;   /* 0: parameter set = KV head h; 1: set = b*Hkv + h                           */
} kv_cache;

size_t kv_cache_bytes(const kv_params* p, int tensor, int B, int Hkv, int64_t T_cap);

/* Encode t_new tokens per sequence (prefill or append).  [AATC; SPECTRA "re-encodes the cache into this
 * coordinate system"]
 *   k, v: device [B][Hkv][t_new][d] in dtype (KV_DTYPE_BF16 or KV_DTYPE_F32), 16-byte aligned;
 *   dst_pos_dev: device int64 [B], token i of sequence b is written at position dst_pos[b] + i, which must
 *   be <= T_cap - t_new (checked on the device: violations are skipped and reported as KV_ERR_DEVICE).
 * Rotation y = T x, then per token y'_j = (y_j - mu_j) * (1/sigma_j), z = fp16(min y'), s = fp16(max y' - z),
 * c_j = clamp(floor(((y'_j - z)/s) * 2^b_j), 0, 2^b_j - 1), packed as above.
 * A value token writes only its own halves (16-bit stores), so a token appended at an odd position leaves
 * the record's earlier token intact.
 * Kernels: bf16 tokens with t_new >= 128 go to the tensor cores (rotation by tcgen05 MMAs against the bf16
 * three-way split of T, fp32 accumulation); fp32 tokens and short appends to CUDA cores (fp32 FMAs). The codes
 * of a given rotated vector are identical on every path; the rotations themselves differ by fp32 rounding
 * order, so the paths agree with each other and with the oracle to the end-to-end bar (1 LSB, rare).
 * Asynchronous on `stream`; a following kv_attend_decode on the same stream may begin preparing while the
 * append kernel finishes (programmatic dependent launch), and waits for it before reading any record. */
kv_status kv_encode(const kv_params* p, const kv_cache* cache, const void* k, const void* v, int dtype,
                    int B, int64_t t_new, const int64_t* dst_pos_dev, kv_stream_t stream);

/* Decode attention over the packed cache for one query per head.  [NOVA-KV: decode re-reads the cache
 * every step and is bandwidth-bound; AATC / SPECTRA transform coding]
 *   q: device bf16 [B][Hq][d]; seq_lens_dev: device int32 [B], 1 <= seq_len <= T_cap (0 gives zeros);
 *   out: device fp32 [B][Hq][d]; softmax_scale (alpha) typically 1/sqrt(d).
 *   o_h = sum_t softmax_t(alpha q_h . k^_t) v^_t, k^ = T_K^T y^ with y^_j = mu_j + sigma_j (z + (c_j + 1/2)
 *   s 2^-b_j) for b_j > 0 and mu_j otherwise (v^ likewise). Computed in the rotated bases: each CTA rotates
 *   q for its (sequence, KV head) in its prologue; each split of the tokens maps its partial sum back to the
 *   original basis (T_V^T folded with sigma), and the last split to finish merges the splits with their
 *   softmax weights. One kernel launch, as a programmatic dependant of the previous kernel of the stream (an
 *   append, say): it reads q and the records only after that kernel has completed.
 *   Arithmetic: each code enters an fp16 tensor-core MMA exactly, as 1 + c 2^-w (w: its slot's width), and the
 *   affine terms of the dequantisation are folded into per-head constants; q's coefficients (scaled per head
 *   by a power of two so that they stay clear of fp16 subnormals) are carried as fp16 hi + lo pairs, p s_V
 *   likewise; each 32-token product sum starts from zero and the running sums are kept in fp32 with
 *   round-to-nearest arithmetic; the softmax runs in base 2 on the hardware exponential. Result: within 2e-3
 *   relative L2 of the exact decode of the same records.
 *   workspace: device, at least kv_decode_workspace_bytes(...) bytes, 16-byte aligned, zero-filled before its
 *   first use (it holds one arrival counter per (sequence, KV head), which every call leaves at zero, so the
 *   workspace is reused across calls without clearing); calls that share a workspace must not overlap on the
 *   device. */
size_t kv_decode_workspace_bytes(const kv_params* p, int B, int Hkv, int Hq, int64_t T_cap);
kv_status kv_attend_decode(const kv_params* p, const kv_cache* cache, const void* q, int B, int Hq,
                           const int32_t* seq_lens_dev, float softmax_scale, float* out,
                           void* workspace, size_t ws_bytes, kv_stream_t stream);

/* Decode attention without a caller-provided workspace. No page has a counterpart; this entry point serves
 * callers that cannot allocate device memory around the call: a serving engine whose memory planner owns
 * all of the GPU's memory and hands a kernel library only pointers and a stream, or code that runs inside an
 * allocator or memory-pool callback, where calling cudaMalloc would re-enter the allocator.
 *   Same arguments, results and errors as kv_attend_decode, minus workspace and ws_bytes: the split
 *   partials, q operands and arrival counters live in one static device array of KV_NOALLOC_SCRATCH_BYTES
 *   bytes compiled into the library (every GPU that loads the library holds it until the process exits).
 *   A shape whose workspace (kv_decode_workspace_bytes) exceeds that size is rejected with
 *   KV_ERR_INVALID_ARG before any launch. The call allocates nothing: no cudaMalloc, cudaFree or
 *   allocating library routine.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that device
 *   current; make that first call before any stream capture.
 *   Every call shares the one array and leaves its contents behind. The array starts zeroed (static device
 *   storage) and every call leaves the arrival counters in it at zero, which is the state the next call
 *   needs; the split partials are written before they are read. Calls whose kernels overlap on the GPU (other
 *   streams, other host threads) race on the array: serialise them. */
#define KV_NOALLOC_SCRATCH_BYTES (4u << 20)
kv_status kv_attend_decode_noalloc(const kv_params* p, const kv_cache* cache, const void* q, int B, int Hq,
                                   const int32_t* seq_lens_dev, float softmax_scale, float* out,
                                   kv_stream_t stream);

/* ------------------------------------------------------------------------------------------------------
 * Paged, multi-layer cache (device, caller-owned).  [SPECTRA abstract: longer contexts and larger batches]
 * Records as in kv_cache, kept in fixed-size pages of page_tokens tokens of one KV head:
 *   k_pages: [n_pages][Hkv][page_tokens][r_words_k]; v_pages: [n_pages][Hkv][page_tokens / 2][2 r_words_v].
 * The view holds n_layers layers of B sequences; virtual sequence z = l * B + b (layer l, sequence b) finds the
 * page of its tokens [i P, (i + 1) P) at block_table[z * max_pages + i] (device int32; only the pages below a
 * sequence's length are read or written). Layer l of the view uses the parameter sets of layer first_layer + l:
 * sets (first_layer + l) * S + (per_seq_params ? b * Hkv + h : h), S = per_seq_params ? B * Hkv : Hkv; so a
 * table calibrated over every layer's heads (layer-major) serves a whole model, and a view of one layer
 * (n_layers = 1, first_layer = l, the block table's rows of that layer) serves one layer at a time.
 * ------------------------------------------------------------------------------------------------------ */
typedef struct {
  uint32_t* k_pages;           /* 16-byte aligned                                                             */
  uint32_t* v_pages;           /* 16-byte aligned                                                             */
  int64_t n_pages;             /* pages in each pool; block-table entries outside 0..n_pages-1 are reported as
                                  KV_ERR_DEVICE by kv_check_status and their tokens are left out (or unwritten) */
  int page_tokens;             /* tokens per page: a power of two from 32 to 2^20                             */
  int Hkv;
  int B;                       /* sequences per layer                                                         */
  int n_layers;                /* layers in the view (>= 1)                                                   */
  int max_pages;               /* block-table row length (pages per sequence); max_pages * page_tokens < 2^31 */
  const int32_t* block_table;  /* device [n_layers * B][max_pages]                                            */
  int per_seq_params;
  int first_layer;             /* parameter layer of the view's layer 0                                       */
} kv_paged_cache;

size_t kv_paged_cache_bytes(const kv_params* p, int tensor, int64_t n_pages, int page_tokens, int Hkv);

/* Encode into a paged cache: as kv_encode, for every layer of the view in one launch.
 *   k, v: device [n_layers][B][Hkv][t_new][d] in dtype; dst_pos_dev: device int64 [B] (the same positions in
 *   every layer); token i of (layer l, sequence b) goes to position dst_pos[b] + i of virtual sequence l B + b,
 *   which must lie below max_pages * page_tokens (checked on the device: violations and bad page indices are
 *   skipped and reported as KV_ERR_DEVICE). Same kernels and codes as kv_encode. */
kv_status kv_encode_paged(const kv_params* p, const kv_paged_cache* cache, const void* k, const void* v,
                          int dtype, int64_t t_new, const int64_t* dst_pos_dev, kv_stream_t stream);

/* Decode attention over a paged cache for every layer of the view in one launch.
 *   q: device bf16 [n_layers][B][Hq][d]; out: device fp32 [n_layers][B][Hq][d]; seq_lens_dev: device int32 [B]
 *   (shared by the layers, 1 <= seq_len <= max_pages * page_tokens, 0 gives zeros).
 *   q_pos_dev: device int32 [B], the position of each sequence's query for the rotary embedding set by
 *   kv_params_set_rope (q is embedded in the kernel's prologue, before the rotation into the key basis), or NULL
 *   when q arrives embedded. Otherwise the same results, precision and conventions as kv_attend_decode: the
 *   records of virtual sequence z stream page by page into the same split-K decode kernel.
 *   workspace: at least kv_decode_paged_workspace_bytes(...) bytes, 16-byte aligned, zero-filled before its
 *   first use and reusable across calls that do not overlap on the device. */
size_t kv_decode_paged_workspace_bytes(const kv_params* p, const kv_paged_cache* cache, int Hq);
kv_status kv_attend_decode_paged(const kv_params* p, const kv_paged_cache* cache, const void* q, int Hq,
                                 const int32_t* seq_lens_dev, const int32_t* q_pos_dev, float softmax_scale,
                                 float* out, void* workspace, size_t ws_bytes, kv_stream_t stream);

/* ------------------------------------------------------------------------------------------------------
 * Token-axis allocation, once after the prefill.  [RDKV, "SPHERICAL KV" page, first abstract: each token gets a
 * width from full precision down to zero bits by reverse water-filling over weights taken from the distortion its
 * compression induces on attention]
 * A token's weight is lambda_t = sum_q p_qt^2 over the observation queries q of the KV head's g query heads
 * (p_q = softmax_t(softmax_scale q . k_t) over the T prefill keys): a white error on token t's value moves query
 * q's output by p_qt times it. With one tier above zero bits (the token keeps its whole record, or is evicted),
 * reverse water-filling keeps the `keep` heaviest tokens of each (sequence, KV head). The kept records are then
 * compacted in order into a cache of their own, over which kv_attend_decode runs with seq_len = keep (appends
 * continue at position keep).
 * ------------------------------------------------------------------------------------------------------ */
/* Token weights. q_obs: device bf16 [B][Hq][W][d] observation queries (e.g. the last W prompt positions'
 * queries, rotary-embedded); k: device bf16 [B][Hkv][T][d] prefill keys; weights: device fp32 [B][Hkv][T].
 * Requires (Hq / Hkv) * W <= 128 and B * Hkv * T < 2^31. The contraction runs on the tensor cores (bf16 operands,
 * fp32 accumulation); logits and weights in fp32. workspace: kv_token_weights_workspace_bytes(...) bytes,
 * 16-byte aligned (no zero fill needed). */
size_t kv_token_weights_workspace_bytes(int B, int Hkv, int64_t T);
kv_status kv_token_weights(const void* q_obs, int W, const void* k, int B, int Hkv, int Hq, int64_t T,
                           float softmax_scale, float* weights, void* workspace, size_t ws_bytes,
                           kv_stream_t stream);
/* The kept tokens: keep_idx (device int32 [B][Hkv][keep]) receives, for every (sequence, KV head), the indices of
 * the keep tokens of largest weight in ascending order (equal weights: the earlier tokens kept; zero, negative
 * and NaN weights rank lowest). weights: device fp32 [B][Hkv][T]; 0 <= keep <= T < 2^31. */
kv_status kv_token_select(const float* weights, int B, int Hkv, int64_t T, int64_t keep, int32_t* keep_idx,
                          kv_stream_t stream);
/* Compaction: token i < keep of (b, h) in dst becomes token keep_idx[b][h][i] of src (records copied; value tokens
 * re-paired two per record, a missing second token's halves 0). src and dst: distinct dense caches of this
 * table's record lengths with the same Hkv; keep <= dst T_cap; indices outside src's T_cap are skipped and
 * reported as KV_ERR_DEVICE. KV_ERR_UNSUPPORTED when B * Hkv > 65535 or one head's kept records exceed 2^31 - 256
 * words. */
kv_status kv_cache_compact(const kv_params* p, const kv_cache* src, const kv_cache* dst, int B,
                           const int32_t* keep_idx, int64_t keep, kv_stream_t stream);

/* Uncompressed bf16 split-K flash-decode over k, v: device bf16 [B][Hkv][T_cap][d]; same q, seq_lens,
 * out conventions. The measurement comparator for the packed path (no page counterpart beyond the
 * full-cache FlashAttention-2 decoding that RDKV compares against). workspace: device, at least
 * kv_decode_bf16_workspace_bytes(...) bytes, 16-byte aligned, zero-filled before its first use (its arrival
 * counters are left at zero by every call); calls sharing a workspace must not overlap on the device. */
size_t kv_decode_bf16_workspace_bytes(int B, int Hkv, int Hq, int64_t T_cap);
kv_status kv_attend_decode_bf16(const void* k, const void* v, int B, int Hkv, int Hq, int64_t T_cap,
                                const void* q, const int32_t* seq_lens_dev, float softmax_scale,
                                float* out, void* workspace, size_t ws_bytes, kv_stream_t stream);

/* Synchronise the stream and return (and clear) the device status word of the current device:
 * KV_OK, KV_ERR_TIMEOUT or KV_ERR_DEVICE; KV_ERR_CUDA if the stream reports an error. */
kv_status kv_check_status(kv_stream_t stream);
const char* kv_last_error(void);
int kv_version(void);

/* ------------------------------------------------------------------------------------------------------
 * Parity and test entry points (same kernels' device code; no separate math).
 * ------------------------------------------------------------------------------------------------------ */
/* Quantise + pack n rotated fp32 vectors y_dev [n][d] (storage order) of one set/tensor into rec_dev (keys:
 * [n][r_words]; values: [ceil(n/2)][2 r_words], a missing second token's half left as it was), running the
 * encode kernels' quantiser. variant 0: warp-per-token (CUDA-core encode); variant 1: thread-per-token;
 * variant 2: the tensor-core encode's epilogue (coefficients staged in tensor memory, reciprocal quotient with the
 * exact redo of near-ties), 128 tokens per CTA. */
kv_status kv_debug_quantize_pack(const kv_params* p, int set, int tensor, const float* y_dev, int64_t n,
                                 uint32_t* rec_dev, int variant, kv_stream_t stream);
/* Run the decoder's slot extraction over the records of n tokens (keys [n][r_words], values
 * [ceil(n/2)][2 r_words]) of one set/tensor and write codes_dev [n][d] (uint16, storage order; 0 for
 * zero-width channels). */
kv_status kv_debug_unpack(const kv_params* p, int set, int tensor, const uint32_t* rec_dev, int64_t n,
                          uint16_t* codes_dev, kv_stream_t stream);
/* Host water-filling used by kv_calibrate: integer widths for importances lam [d] and budget bits. */
kv_status kv_debug_water_fill(const double* lam, int d, int budget_bits, int max_bits, int32_t* widths);
/* Host Jacobi eigensolver used by kv_calibrate: sym [d][d] -> eigenvalues descending [d] and eigenvectors
 * as columns evecs [d][d] (row-major), sign-normalised. */
kv_status kv_debug_eigh(const double* sym, int d, double* evals, double* evecs);
/* Encode path selection for tests: 0 automatic (bf16 with at least 128 new tokens per head: tensor cores;
 * otherwise CUDA cores), 1 CUDA cores (one CTA per head for up to 16 new tokens, else one warp per token; the
 * two write identical records), 2 tensor-core tiles (bf16 only; KV_ERR_UNSUPPORTED for fp32). */
kv_status kv_debug_set_encode_path(int path);
/* Device wait limit in nanoseconds for the bounded mbarrier waits (default 2e9). */
kv_status kv_debug_set_wait_limit_ns(long long ns);
/* Launch a kernel that waits on an mbarrier nothing will complete, with the current wait limit; it must
 * return, leaving KV_ERR_TIMEOUT for kv_check_status. */
kv_status kv_debug_wait_timeout_selftest(kv_stream_t stream);
/* The launch kv_attend_decode would make for these parameters and shapes on the current device, without
 * launching: info[12] = cluster size (0: the splits merge through the workspace), splits per (sequence, KV
 * head), ring stages, warps per CTA, 16-channel blocks, dynamic shared memory bytes, then the clusters the
 * device holds at once for cluster sizes 16, 8, 4, 2, 1 (-1: size not considered), then 1 when the kernel takes
 * every channel block's codes in one shared-memory load per lane (each lane's two slots share a code word in all
 * blocks of all sets), else 0. Host memory. */
kv_status kv_debug_decode_plan(const kv_params* p, int B, int Hkv, int Hq, int64_t T_cap, int32_t* info);

#ifdef __cplusplus
}
#endif
#endif /* KVTC_H */
