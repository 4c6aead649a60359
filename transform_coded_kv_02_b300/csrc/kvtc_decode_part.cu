// One part of the decode kernel's compiled variants (decode_kernel and its launcher, kvtc_decode.cuh). The file is
// compiled once per part number (-DKVTC_DECODE_PART=0 .. DECODE_PARTS - 1) into separate translation units, so
// that the variants build in parallel; kvtc_kernels.cu dispatches to them. Each unit has its own device status
// word, which read_and_clear_decode_status reads for kv_check_status.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdio.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "kvtc_codec.cuh"
#include "kvtc_internal.h"
#include "kvtc_launch.cuh"
#include "kvtc_ptx.cuh"

#ifndef KVTC_DECODE_PART
#error "compile with -DKVTC_DECODE_PART=<part number>"
#endif
#define KVTC_DECODE_KERNELS
#include "kvtc_decode.cuh"

namespace kvtc {

// explicit instantiation of one launcher variant (and so of its two kernels, cluster and workspace merge)
#define KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)                                                 \
  template cudaError_t launch_decode_kernel<NB, RK, RV, NBLK, NW, SW>(cudaLaunchConfig_t&, const ParamsDev&,  \
                                                                       DecArgs, int, int32_t*);
#if KVTC_DECODE_PART == 0
#define KVTC_DECODE_IN_PART_0(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_0(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 1
#define KVTC_DECODE_IN_PART_1(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_1(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 2
#define KVTC_DECODE_IN_PART_2(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_2(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 3
#define KVTC_DECODE_IN_PART_3(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_3(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 4
#define KVTC_DECODE_IN_PART_4(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_4(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 5
#define KVTC_DECODE_IN_PART_5(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_5(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 6
#define KVTC_DECODE_IN_PART_6(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_6(NB, RK, RV, NBLK, NW, SW)
#endif
#if KVTC_DECODE_PART == 7
#define KVTC_DECODE_IN_PART_7(NB, RK, RV, NBLK, NW, SW) KVTC_DECODE_INSTANTIATE(NB, RK, RV, NBLK, NW, SW)
#else
#define KVTC_DECODE_IN_PART_7(NB, RK, RV, NBLK, NW, SW)
#endif
#define KVTC_DECODE_IN_PART(NB, RK, RV, NBLK, NW, SW, PART) KVTC_DECODE_IN_PART_##PART(NB, RK, RV, NBLK, NW, SW)

KVTC_DECODE_VARIANTS(KVTC_DECODE_IN_PART)

#define KVTC_CAT2(a, b) a##b
#define KVTC_CAT(a, b) KVTC_CAT2(a, b)

// this part's status word
static kv_status read_and_clear_status_here(unsigned* out) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  if (e != cudaSuccess) {
    set_error("device status (decode part %d): %s", KVTC_DECODE_PART, cudaGetErrorString(e));
    return KV_ERR_CUDA;
  }
  *out = v;
  return KV_OK;
}
kv_status KVTC_CAT(read_and_clear_decode_status_, KVTC_DECODE_PART)(unsigned* out) {
  return read_and_clear_status_here(out);
}

}  // namespace kvtc
