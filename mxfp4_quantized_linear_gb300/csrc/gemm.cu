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
// The producer requests its first unit's weight stages before the grid
// dependency wait (the weight does not depend on the quantizer before it).
// When the tiles would leave more than half the SMs idle (M of a few hundred
// rows on a narrow N), K is split into ranges: one (tile, range) unit a CTA,
// its f32 sums staged through the idle operand ring into the workspace, and
// gemm_finish_kernel adds a tile's ranges in order, the bias, and rounds once.
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
  int ksplit;                 // K ranges a tile (gemm_ksplit); > 1: f32 partial sums to part
  float* part;                // [ksplit, M, N]
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
  // work units: (tile, K range), the range fastest
  const int S = p.ksplit;
  const int nunits = p.m_tiles * p.n_tiles * S;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&bmap);
    const uint64_t pol_a = policy_evict_last(), pol_b = policy_evict_last();
    // a stage's weight half: B and its two scale atoms
    auto load_b = [&](int stage, int kt, int nt) {
      uint8_t* st = smem + stage * kStageBytes;
      const int rb0 = min(2 * nt, p.RTb - 1), rb1 = min(2 * nt + 1, p.RTb - 1);
      tma_load_2d(st + kABytes, &bmap, &full[stage], kt * BKB, nt * BN, pol_b);
      bulk_load(st + kABytes + kBBytes + kSfaBytes, p.sfb + (static_cast<long long>(rb0) * p.KT + kt) * 512, 512,
                &full[stage]);
      bulk_load(st + kABytes + kBBytes + kSfaBytes + 512, p.sfb + (static_cast<long long>(rb1) * p.KT + kt) * 512,
                512, &full[stage]);
    };
    // the weights do not depend on the kernel before (the activation
    // quantizer): the first unit's first stages start loading them before the
    // dependency wait, so they stream while the quantizer finishes (each
    // stage's barrier expects its activation half too)
    int pre = 0;
    if (static_cast<int>(blockIdx.x) < nunits) {
      const int tile = blockIdx.x / S, ks = blockIdx.x - tile * S;
      const int k0 = ks * p.KT / S, k1 = (ks + 1) * p.KT / S;
      pre = min(kStages, k1 - k0);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], kTxBytes);  // stage i is free: nothing has used it yet
        load_b(i, k0 + i, tile / p.m_tiles);
      }
    }
    pdl_wait_prior_grid();  // the quantized activation is complete and visible
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x) {
      const int tile = u / S, ks = u - tile * S;
      const int mt = tile % p.m_tiles, nt = tile / p.m_tiles;
      const int k0 = ks * p.KT / S;
      for (int kt = k0; kt < (ks + 1) * p.KT / S; ++kt) {
        const bool early = u == static_cast<int>(blockIdx.x) && kt - k0 < pre;  // weight half already loading
        if (!early) {
          if (!mbar_wait(&empty[stage], phase ^ 1u)) { *abort_flag = 1u; break; }
          mbar_arrive_expect_tx(&full[stage], kTxBytes);
          load_b(stage, kt, nt);
        }
        uint8_t* st = smem + stage * kStageBytes;
        tma_load_2d(st, &amap, &full[stage], kt * BKB, mt * BM, pol_a);
        bulk_load(st + kABytes + kBBytes, p.sfa + (static_cast<long long>(mt) * p.KT + kt) * 512, 512, &full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x) {
      const int ks = u % S, k0 = ks * p.KT / S, k1 = (ks + 1) * p.KT / S;
      if (!mbar_wait(acc_empty, acc_phase ^ 1u)) { *abort_flag = 1u; break; }
      tc_fence_after();
      for (int kt = k0; kt < k1; ++kt) {
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
                      (kt != k0 || k != 0) ? 1u : 0u);
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
    for (int u = blockIdx.x; u < nunits && !*abort_flag; u += gridDim.x) {
      const int tile = u / S, ks = u - tile * S;
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
      if (S > 1) {
        // this K range's f32 sums; the finishing kernel adds the ranges and the
        // bias.  A split grid runs one unit a CTA, so the operand ring is idle
        // once the accumulator is full: each warp transposes its 32 rows x 128
        // columns through 16.5 KB of it (rows padded to 132 words) and stores
        // whole rows, a warp 512 contiguous bytes an instruction.
        float* stg = reinterpret_cast<float*>(smem) + (warp - 2) * 32 * 132;
#pragma unroll
        for (int j = 0; j < 128; j += 4)
          *reinterpret_cast<float4*>(stg + lane * 132 + j) =
              make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                          __uint_as_float(r[j + 3]));
        __syncwarp();
        const int row0 = mt * BM + q * 32;
        const int rows = min(32, p.M - row0);
        const bool vec = (p.N & 3) == 0 && nb + lane * 4 + 4 <= p.N;
        for (int rr = 0; rr < rows; ++rr) {
          const float4 v = *reinterpret_cast<const float4*>(stg + rr * 132 + lane * 4);
          float* dst = p.part + (static_cast<long long>(ks) * p.M + row0 + rr) * p.N + nb + lane * 4;
          if (vec) {
            *reinterpret_cast<float4*>(dst) = v;
          } else {
            const float e[4] = {v.x, v.y, v.z, v.w};
            for (int c = 0; c < 4; ++c)
              if (nb + lane * 4 + c < p.N) dst[c] = e[c];
          }
        }
      } else if (row < p.M) {
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

// Split-K finish: out[m, n] = bf16(sum over the S ranges of part[s, m, n], in
// range order, + bias[n]); one thread a 4 consecutive columns of a row.
// Launched as a programmatic dependent of the GEMM.
__global__ void __launch_bounds__(256) gemm_finish_kernel(const float* __restrict__ part, int S, int M, int N,
                                                          const __nv_bfloat16* __restrict__ bias,
                                                          __nv_bfloat16* __restrict__ out) {
  pdl_wait_prior_grid();
  const int N4 = (N + 3) >> 2;
  const long long total = static_cast<long long>(M) * N4;
  const long long plane = static_cast<long long>(M) * N;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i / N4), n = static_cast<int>(i - static_cast<long long>(m) * N4) * 4;
    const float* src = part + static_cast<long long>(m) * N + n;
    if (n + 4 <= N && (N & 3) == 0) {
      float4 v = *reinterpret_cast<const float4*>(src);
      for (int k = 1; k < S; ++k) {
        const float4 w = *reinterpret_cast<const float4*>(src + k * plane);
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
      }
      if (bias) {
        v.x += __bfloat162float(bias[n]);
        v.y += __bfloat162float(bias[n + 1]);
        v.z += __bfloat162float(bias[n + 2]);
        v.w += __bfloat162float(bias[n + 3]);
      }
      const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&a);
      pk.y = *reinterpret_cast<const uint32_t*>(&b);
      *reinterpret_cast<uint2*>(out + static_cast<long long>(m) * N + n) = pk;
    } else {
      for (int c = 0; c < 4 && n + c < N; ++c) {
        float v = src[c];
        for (int k = 1; k < S; ++k) v += src[k * plane + c];
        if (bias) v += __bfloat162float(bias[n + c]);
        out[static_cast<long long>(m) * N + n + c] = __float2bfloat16_rn(v);
      }
    }
  }
}

}  // namespace

unsigned int take_error_flags_gemm() { return take_tu_error_flags(); }

// K ranges a tile: only when the 128 x 256 tiles would leave more than half
// the SMs idle (M up to a few hundred rows on a narrow N); then enough ranges
// to fill one wave, at most 8, each of at least 4 K steps, with at most 64 MB
// of partial sums -- and no more than `room` bytes of them.  (N=7168 K=8192:
// 28 tiles at M = 64 / 128 leave 124 of 152 SMs idle.)
int gemm_ksplit(int M, int N, int Kp, int sms, size_t room) {
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN), KT = Kp / BKB;
  if (tiles <= 0 || 2 * tiles > sms) return 1;
  int S = sms / tiles;
  if (S > 8) S = 8;
  if (S > KT / 4) S = KT / 4;
  const size_t plane = static_cast<size_t>(M) * static_cast<size_t>(N) * 4;
  const size_t cap = room < (static_cast<size_t>(64) << 20) ? room : (static_cast<size_t>(64) << 20);
  while (S > 1 && S * plane > cap) --S;
  return S > 1 ? S : 1;
}

size_t gemm_part_bytes(int M, int N, int Kp, int sms) {
  const int S = gemm_ksplit(M, N, Kp, sms, ~static_cast<size_t>(0));
  return S > 1 ? static_cast<size_t>(S) * M * static_cast<size_t>(N) * 4 : 0;
}

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
  p.ksplit = a.part ? gemm_ksplit(a.M, w->N, w->Kp, di.sm_count, a.part_bytes) : 1;
  p.part = static_cast<float*>(a.part);
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
  const int nunits = p.m_tiles * p.n_tiles * p.ksplit;
  const int grid = nunits < di.sm_count ? nunits : di.sm_count;
  // the split epilogue stages its stores in the operand ring: one unit a CTA
  if (p.ksplit > 1 && nunits > grid) return set_error(MX_ERR_UNSUPPORTED, "K split of %d units on %d CTAs", nunits, grid);
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
  if (p.ksplit > 1) {
    const long long items = static_cast<long long>(a.M) * ((w->N + 3) / 4);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks_for(items, 256)), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, gemm_finish_kernel, static_cast<const float*>(p.part), p.ksplit, a.M, w->N,
                           p.bias, p.out);
    if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "gemm finish launch: %s", cudaGetErrorString(e));
  }
  return MX_OK;
}

}  // namespace mx
