// sm_103a kernels of the transform-coded KV cache and their launchers: this CUDA translation unit, made of
//  kvtc_encode.cuh     encode_warp_kernel: one warp per (tensor, sequence, head, token); y = T x with CUDA-core
//                      FMAs, then the warp quantiser/packer (append and fp32 inputs)
//  kvtc_encode_tc.cuh  encode_tc_kernel: 128-token tiles staged by TMA, y = X T^T on the tensor cores (tcgen05,
//                      split-bf16 T, fp32 accumulators in tensor memory), thread-per-token quantiser/packer
//  kvtc_decode.cuh     the decode's split plan, workspace layout and dispatch; decode_kernel itself (split-K
//                      flash-decode over the packed records: q' and the folded logit constants in the prologue,
//                      bulk-copy ring, codes unpacked straight into warp-MMA operands, logits, softmax and P.V in
//                      every warp, split merge in a cluster or through the workspace) is compiled in the
//                      kvtc_decode_part.cu units
//  kvtc_bf16.cuh       decode_bf16_kernel: the same split-K structure over an uncompressed bf16 cache
//  kvtc_token.cuh      token-axis allocation: token weights from the observation queries' attention (tcgen05),
//                      the kept tokens per (sequence, KV head), record compaction
//  kvtc_debug.cuh      parity and self-test kernels behind the kv_debug_* entry points
//
// Method sources: "KV Cache Compression Through the Lens of Transform Coding" (AATC), Key points;
// "SPECTRA ..." abstract; "SPHERICAL KV ..." page, third abstract (NOVA-KV: decode reads the cache every step
// and is bandwidth-bound; reconstruction must stay cheap).
//
// Decode algebra (rotated domain). With y^_j = mu_j + sigma_j (z + (c_j + 1/2) s 2^-b_j) for b_j > 0:
//   a q.k^ = a (T q).y^ = C0 + z C1 + s sum_{b_j>0} q'_j (c_j + 1/2)
//   sum_t p_t v^_t = T_V^T o^,  o^_j = mu_j + sigma_j (Z + 2^-b_j A_j) / l for b_j > 0 (mu_j otherwise),
//   Z = sum_t p_t z_t, A_j = sum_t p_t s_t (c_tj + 1/2), l = sum_t p_t;
// kvtc_decode.cuh states the form the kernel evaluates (codes entering the MMA as 1 + c 2^-w).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "kvtc_codec.cuh"
#include "kvtc_internal.h"
#include "kvtc_launch.cuh"
#include "kvtc_ptx.cuh"

namespace kvtc {

static long long g_wait_limit_ns = 2000000000LL;

void set_wait_limit_ns(long long ns) { g_wait_limit_ns = ns; }

static kv_status launch_check(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

// the decode parts' status readers (kvtc_decode_part.cu)
kv_status read_and_clear_decode_status_0(unsigned* out);
kv_status read_and_clear_decode_status_1(unsigned* out);
kv_status read_and_clear_decode_status_2(unsigned* out);
kv_status read_and_clear_decode_status_3(unsigned* out);
kv_status read_and_clear_decode_status_4(unsigned* out);
kv_status read_and_clear_decode_status_5(unsigned* out);
kv_status read_and_clear_decode_status_6(unsigned* out);
kv_status read_and_clear_decode_status_7(unsigned* out);
static_assert(DECODE_PARTS == 8, "one status reader per decode part");

kv_status read_and_clear_decode_status(int part, unsigned* out) {
  using Reader = kv_status (*)(unsigned*);
  static const Reader readers[DECODE_PARTS] = {
      read_and_clear_decode_status_0, read_and_clear_decode_status_1, read_and_clear_decode_status_2,
      read_and_clear_decode_status_3, read_and_clear_decode_status_4, read_and_clear_decode_status_5,
      read_and_clear_decode_status_6, read_and_clear_decode_status_7};
  if (part < 0 || part >= DECODE_PARTS) {
    set_error("decode part %d out of range", part);
    return KV_ERR_INVALID_ARG;
  }
  return readers[part](out);
}

// the status word of this translation unit, then those of the decode parts
kv_status read_and_clear_device_status(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  if (e != cudaSuccess) {
    set_error("device status: %s", cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  for (int part = 0; part < DECODE_PARTS; ++part) {
    unsigned pv = 0;
    const kv_status st = read_and_clear_decode_status(part, &pv);
    if (st != KV_OK) return st;
    v |= pv;
  }
  *out = v;
  return KV_OK;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace kvtc

#include "kvtc_encode_tc.cuh"
#include "kvtc_encode.cuh"
#include "kvtc_decode.cuh"
#include "kvtc_bf16.cuh"
#include "kvtc_token.cuh"
#include "kvtc_debug.cuh"

namespace kvtc {

// ======================================================================================================
// decode with the library's own fixed scratch (no allocation on the call path)
// ======================================================================================================
// The scratch array. Host code must not use its name as an address (on the host it is only a stand-in);
// the device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KV_NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[NOALLOC_MAX_DEVICES] = {};

// dev: the current device (the lookup must run with it current)
static kv_status noalloc_scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
    set_error("device %d beyond the %d devices the static scratch table covers", dev, NOALLOC_MAX_DEVICES);
    return KV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      set_error("cudaGetSymbolAddress(static scratch) on device %d: %s", dev, cudaGetErrorString(e));
      return KV_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return KV_OK;
}

}  // namespace kvtc

extern "C" kv_status kv_attend_decode_noalloc(const kv_params* p, const kv_cache* c, const void* q, int B, int Hq,
                                              const int32_t* seq_lens_dev, float softmax_scale, float* out,
                                              kv_stream_t stream) {
  kvtc::clear_error();
  int dev = 0;
  kv_status st = kvtc::check_decode_args(p, c, q, B, Hq, seq_lens_dev, softmax_scale, out, &dev);
  if (st != KV_OK) return st;
  const kvtc::DecodeLayout L = kvtc::decode_layout(B, c->Hkv, Hq, c->T_cap, dev);
  if (L.total > (size_t)KV_NOALLOC_SCRATCH_BYTES) {
    kvtc::set_error("decode of B=%d Hkv=%d T_cap=%lld needs %zu bytes of scratch, more than the library's fixed "
                    "%u bytes; use kv_attend_decode with a workspace", B, c->Hkv, (long long)c->T_cap, L.total,
                    (unsigned)KV_NOALLOC_SCRATCH_BYTES);
    return KV_ERR_INVALID_ARG;
  }
  void* ws = nullptr;
  if ((st = kvtc::noalloc_scratch_address(dev, &ws)) != KV_OK) return st;
  return kvtc::launch_decode(p->dev, kvtc::dense_view(*c), q, B, Hq, seq_lens_dev, nullptr, softmax_scale, out, ws,
                             L, (cudaStream_t)stream);
}

