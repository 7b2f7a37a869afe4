// K-GEMM: block-scaled MXFP8 GEMM for large M on the 5th-generation tensor cores.
//
// out[m, n] = sum_k xq[m, k] W[n, k] 2^(cx[m, k/32] - 127) 2^(cw[n, k/32] - 127)
// (rocm_native = vllm.model_executor.kernels.linear.mxfp8.rocm_native, _launch:
// out = x @ w.T, x MXFP8-quantized per token, weight 32x32 block scales expanded
// per row at pack time).  The page's gfx950 path tiles M=4096 prefill with
// 128x128x256 dot_scaled tiles (_select_cfg); here the scales are applied by the
// tensor core itself: `tcgen05.mma ... kind::mxf8f6f4.block_scale.scale_vec::1X`
// with one E8M0 code per row per 32-wide K block held in tensor memory.
//
// CTA = 10 warps, one CTA per SM, persistent over 128 x 256 output tiles:
//   warp 0 (lane 0)  TMA producer: per 128-byte K step, A 128x128 and B 256x128
//                    boxes (128B swizzle) plus the 512-byte scale-factor atoms of
//                    A (1) and B (2), all completing on one mbarrier;
//   warp 1 (lane 0)  MMA issuer: copies the step's scale factors into tensor
//                    memory (tcgen05.cp .32x128b.warpx4) and issues 4 MMAs of
//                    K = 32 (scale-factor id k picks byte k of each code word),
//                    accumulating 128 x 256 f32 in tensor memory; tcgen05.commit
//                    frees the smem stage and, after the last step, signals the
//                    epilogue;
//   warps 2..9       epilogue, two warps per tensor-memory lane quarter, 128
//                    columns each: tcgen05.ld of the warp's 32 rows x 128
//                    columns into registers, release of the accumulator (the
//                    next tile's MMAs start), then bias in f32, bf16 round and
//                    store from registers, overlapping those MMAs.
// Every mbarrier wait is bounded; on a timeout the CTA flags the error, stops
// issuing, and still frees its tensor memory.

#include "mx_common.cuh"
#include "mx_internal.h"
#include "tc_common.cuh"

namespace mx {
namespace {

constexpr int BM = 128, BN = 256, BKB = 128;      // tile rows, tile cols, K bytes a step
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kABytes = BM * BKB;                  // 16 KB
constexpr int kBBytes = BN * BKB;                  // 32 KB
constexpr int kSfaBytes = 512, kSfbBytes = 1024;
constexpr int kStageBytes = 51200;                 // A | B | SFA | SFB, rounded to 1024
constexpr int kTxBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                    // 256 f32 columns
constexpr uint32_t kSfCol = 256;                   // + 16 columns a stage: SFA 4, SFB 8
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;

struct GemmParams {
  const uint8_t* sfa;         // activation scale atoms [Mp/128][KT][512]
  const uint8_t* sfb;         // weight scale atoms [ceil(N/128)][KT][512]
  const __nv_bfloat16* bias;  // [N] or null
  __nv_bfloat16* out;         // [M, N]
  int M, N, KT, RTb, m_tiles, n_tiles;
};

constexpr uint32_t kIdesc = mxf8_idesc(BM, BN);

__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap amap,
                                                           const __grid_constant__ CUtensorMap bmap,
                                                           const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    *abort_flag = 0u;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // only now that this CTA holds its tensor memory: a dependent grid then
  // never takes columns that a CTA of this grid still waits for
  pdl_launch_dependents();
  const int ntiles = p.m_tiles * p.n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&bmap);
    const uint64_t pol_a = policy_evict_last(), pol_b = policy_evict_last();
    pdl_wait_prior_grid();  // the quantized activation is complete and visible
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
      const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
      const int rb0 = min(2 * nt, p.RTb - 1), rb1 = min(2 * nt + 1, p.RTb - 1);
      for (int kt = 0; kt < p.KT; ++kt) {
        if (!mbar_wait(&empty[stage], phase ^ 1u)) { *abort_flag = 1u; break; }
        uint8_t* st = smem + stage * kStageBytes;
        mbar_arrive_expect_tx(&full[stage], kTxBytes);
        tma_load_2d(st, &amap, &full[stage], kt * BKB, mt * BM, pol_a);
        tma_load_2d(st + kABytes, &bmap, &full[stage], kt * BKB, nt * BN, pol_b);
        bulk_load(st + kABytes + kBBytes, p.sfa + (static_cast<long long>(mt) * p.KT + kt) * 512, 512, &full[stage]);
        bulk_load(st + kABytes + kBBytes + kSfaBytes, p.sfb + (static_cast<long long>(rb0) * p.KT + kt) * 512, 512,
                  &full[stage]);
        bulk_load(st + kABytes + kBBytes + kSfaBytes + 512, p.sfb + (static_cast<long long>(rb1) * p.KT + kt) * 512,
                  512, &full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
      if (!mbar_wait(acc_empty, acc_phase ^ 1u)) { *abort_flag = 1u; break; }
      tc_fence_after();
      for (int kt = 0; kt < p.KT; ++kt) {
        if (!mbar_wait(&full[stage], phase)) { *abort_flag = 1u; break; }
        tc_fence_after();
        const uint32_t st = smem_u32(smem + stage * kStageBytes);
        const uint32_t sf_col = tmem + kSfCol + stage * 16;
        tc_cp_sf(sf_col, sf_desc(st + kABytes + kBBytes));
        tc_cp_sf(sf_col + 4, sf_desc(st + kABytes + kBBytes + kSfaBytes));
        tc_cp_sf(sf_col + 8, sf_desc(st + kABytes + kBBytes + kSfaBytes + 512));
        const uint64_t adesc = sw128_desc(st);
        const uint64_t bdesc = sw128_desc(st + kABytes);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t idesc = kIdesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
          // +32 bytes along K inside the swizzle atom = +2 in the start-address field
          tc_mma_mxf8(tmem + kAccCol, adesc + 2 * k, bdesc + 2 * k, idesc, sf_col, sf_col + 4,
                      (kt | k) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      tc_commit(acc_full);
      acc_phase ^= 1u;
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // tensor-memory lane quarter this warp may access
    const int half = (warp - 2) >> 2;    // columns [128 half, 128 half + 128)
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < ntiles && !*abort_flag; tile += gridDim.x) {
      const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
      if (!mbar_wait(acc_full, acc_phase)) { *abort_flag = 1u; break; }
      tc_fence_after();
      uint32_t r[128];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + kAccCol + half * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_async(taddr + c * 32, r + 32 * c);
      tmem_wait_ld();
      // the accumulator is in registers: the next tile's MMAs may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_phase ^= 1u;
      const int row = mt * BM + q * 32 + lane;
      const int nb = nt * BN + half * 128;
      if (row < p.M) {
        __nv_bfloat16* dst = p.out + static_cast<long long>(row) * p.N + nb;
        if (nb + 128 <= p.N && (p.N & 7) == 0) {
#pragma unroll
          for (int j = 0; j < 128; j += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float a = __uint_as_float(r[j + 2 * h]), b = __uint_as_float(r[j + 2 * h + 1]);
              if (p.bias) {
                a += __bfloat162float(p.bias[nb + j + 2 * h]);
                b += __bfloat162float(p.bias[nb + j + 2 * h + 1]);
              }
              const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
              pk[h] = *reinterpret_cast<const uint32_t*>(&v);
            }
            *reinterpret_cast<uint4*>(dst + j) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 128; ++j) {
            if (nb + j < p.N) {
              float a = __uint_as_float(r[j]);
              if (p.bias) a += __bfloat162float(p.bias[nb + j]);
              dst[j] = __float2bfloat16_rn(a);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

unsigned int take_error_flags_gemm() { return take_tu_error_flags(); }

int launch_gemm(const GemmArgs& a, cudaStream_t stream) {
  const mx_packed_weight* w = a.w;
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  GemmParams p = {};
  p.sfa = a.sfa;
  p.sfb = w->sf;
  p.bias = static_cast<const __nv_bfloat16*>(a.bias);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = a.M;
  p.N = w->N;
  p.KT = w->Kp / BKB;
  p.RTb = (w->N + 127) / 128;
  p.m_tiles = (a.M + BM - 1) / BM;
  p.n_tiles = (w->N + BN - 1) / BN;
  const int Mp = p.m_tiles * BM;
  CUtensorMap amap, bmap;
  const uint64_t a_cols = a.xq_cols ? a.xq_cols : w->Kp, a_rows = a.xq_rows ? a.xq_rows : Mp;
  const uint64_t a_ld = a.xq_ld ? a.xq_ld : w->Kp;
  int rc = encode_tensor_map_2d(&amap, a.xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_cols, a_rows, a_ld, BKB, BM,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != MX_OK) return rc;
  rc = encode_tensor_map_2d(&bmap, w->bytes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->Kp, w->N, w->Kp, BKB, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != MX_OK) return rc;
  static int smem_set[64];
  if (raise_smem_limit(reinterpret_cast<const void*>(gemm_kernel), kSmemBytes, di, smem_set) != MX_OK)
    return MX_ERR_CUDA;
  cudaError_t e;
  const int ntiles = p.m_tiles * p.n_tiles;
  const int grid = ntiles < di.sm_count ? ntiles : di.sm_count;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_kernel, amap, bmap, p);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

}  // namespace mx
