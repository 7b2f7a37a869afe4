// Dense MXFP8 tensor peak of this GPU, measured: every SM runs a loop of
// block-scaled tcgen05 MMAs (kind::mxf8f6f4, scale_vec::1X, the instruction the
// GEMM and the expert GEMM issue) on operands already in shared memory, with
// no loads, stores or epilogue.  The result is the denominator for the
// tensor-bound kernels' roofline fraction.
//
// One CTA an SM (all 512 tensor-memory columns), two issuing threads in two
// warps, each with its own 128 x 224 f32 accumulator: one thread issues a
// block-scaled MMA only about every 150 cycles, while an M=128 N=224 K=32 MMA
// takes about 130 cycles of tensor time at the nominal rate, so two issuers
// keep the tensor core busy.  Operands: A 128 x 128 bytes and B 224 x 128
// bytes of e4m3 1.0 (128B-swizzled K-major), all scale codes 127, so every MMA
// adds 32 to each accumulator element; the accumulators are checked after the
// loop.  Every wait is bounded.

#include "mx_common.cuh"
#include "mx_internal.h"
#include "tc_common.cuh"

namespace mx {
namespace {

constexpr int kPeakN = 224;
constexpr uint32_t kPeakIdesc = mxf8_idesc(128, kPeakN);
constexpr int kPeakSmem = 120 * 1024;  // one CTA an SM

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int* bad) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* A = smem;                 // 16 KB: 128 rows x 128 B
  uint8_t* B = smem + 16384;         // 32 KB: 256 rows x 128 B (224 used)
  uint8_t* SF = smem + 49152;        // SFA 512 B, SFB 2 x 512 B
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 50688);  // [0] scale copy, [1] the two issuers
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 50704);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 49152 / 4; i += 128) reinterpret_cast<uint32_t*>(A)[i] = 0x38383838u;  // e4m3 1.0
  for (int i = threadIdx.x; i < 1536 / 4; i += 128) reinterpret_cast<uint32_t*>(SF)[i] = 0x7f7f7f7fu;   // 2^0
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 2);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) tmem_alloc(slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t sfa = tmem + 448, sfb = tmem + 452;
  if (threadIdx.x == 0) {
    tc_cp_sf(sfa, sf_desc(smem_u32(SF)));
    tc_cp_sf(sfb, sf_desc(smem_u32(SF + 512)));
    tc_cp_sf(sfb + 4, sf_desc(smem_u32(SF + 1024)));
    tc_commit(&bar[0]);
    mbar_wait(&bar[0], 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (lane == 0 && warp < 2) {
    const uint32_t acc = tmem + static_cast<uint32_t>(warp * kPeakN);
    const uint64_t adesc = sw128_desc(smem_u32(A)), bdesc = sw128_desc(smem_u32(B));
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t idesc = kPeakIdesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
        tc_mma_mxf8(acc, adesc + 2 * k, bdesc + 2 * k, idesc, sfa, sfb, (it | k) != 0 ? 1u : 0u);
      }
    }
    tc_commit(&bar[1]);
  }
  __syncwarp();
  const bool done = mbar_wait(&bar[1], 0);
  tc_fence_after();
  // column 0 of each accumulator, all 128 lanes: 32 per MMA of the chain
  uint32_t v[16];
  tmem_ld16_async(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
  tmem_wait_ld();
  uint32_t w[16];
  tmem_ld16_async(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kPeakN, w);
  tmem_wait_ld();
  const float want = 32.0f * 4.0f * static_cast<float>(iters);
  if (!done || __uint_as_float(v[0]) != want || __uint_as_float(w[0]) != want) atomicAdd(bad, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

unsigned int take_error_flags_peak() { return take_tu_error_flags(); }

}  // namespace mx

using namespace mx;

extern "C" int mx_measure_mxf8_peak(int iters, int reps, double* tflops, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!tflops) return set_error(MX_ERR_ARG, "NULL output");
  *tflops = 0.0;
  if (iters < 1 || iters > (1 << 16) || reps < 1 || reps > 1000)
    return set_error(MX_ERR_ARG, "iters=%d reps=%d: need 1..65536 and 1..1000", iters, reps);
  DeviceInfo di;
  int rc = current_device_info(&di);
  if (rc != MX_OK) return rc;
  if (di.cc_major != 10 || di.cc_minor != 3)
    return set_error(MX_ERR_UNSUPPORTED, "device compute capability %d.%d is not sm_103", di.cc_major,
                     di.cc_minor);
  static int smem_set[64];
  if (raise_smem_limit(reinterpret_cast<const void*>(mma_peak_kernel), kPeakSmem, di, smem_set) != MX_OK)
    return MX_ERR_CUDA;
  // the accumulator check counts into this unit's device error word (no
  // allocation); a bounded wait that times out sets it too
  int* bad = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&bad), g_error_flags);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "peak: %s", cudaGetErrorString(e));
  cudaEvent_t e0, e1;
  if ((e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess)
    return set_error(MX_ERR_CUDA, "peak: events: %s", cudaGetErrorString(e));
  const dim3 grid(di.sm_count), block(128);
  // one launch to warm up, then `reps` launches back to back between the events
  mma_peak_kernel<<<grid, block, kPeakSmem, stream>>>(iters, bad);
  cudaEventRecord(e0, stream);
  for (int r = 0; r < reps; ++r) mma_peak_kernel<<<grid, block, kPeakSmem, stream>>>(iters, bad);
  cudaEventRecord(e1, stream);
  e = cudaEventSynchronize(e1);
  float ms = 0.0f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "peak: %s", cudaGetErrorString(e));
  const unsigned int flags = take_error_flags_peak();
  if (flags & 0x80000000u) return set_error(MX_ERR_CUDA, "peak: could not read the check word");
  if (flags != 0) return set_error(MX_ERR_TIMEOUT, "peak: accumulators wrong or a wait timed out (%u)", flags);
  const double flops = 2.0 * 128.0 * kPeakN * 32.0 * 4.0 * 2.0 * iters * di.sm_count * reps;
  *tflops = flops / (static_cast<double>(ms) * 1e-3) / 1e12;
  return MX_OK;
}
