// K-GEMV: split-K MXFP8 x MXFP8 linear for decode (M <= 32 tokens).
//
// out = x @ w^T (rocm_native = vllm.model_executor.kernels.linear.mxfp8.rocm_native,
// _launch), with the bf16 activation MXFP8-quantized per token inside the call
// (rocm_native, apply_weights / _quant_mxfp8_tile) and every 32-wide K block
// scaled by 2^(cw - 127) * 2^(cx - 127).  The page's decode tiles are narrow
// in N with long K steps because tiny-M GEMV is bound by weight bandwidth and
// by how many compute units stream it (rocm_native, _select_cfg); here that
// becomes: every CTA streams a 64-row x K-slice of the weight through TMA, and
// the CTAs of one row tile split K and reduce through distributed shared memory.
//
// Structure of one CTA (4 warps, 64 weight rows, one K slice):
//   - each warp owns 16 rows and its own NSTAGE-deep ring of 16x128-byte TMA
//     boxes (128B swizzle), refilled by its lane 0 as soon as a stage is used;
//   - the activation slice (<= 32 tokens) sits in shared memory as e4m3 bytes
//     plus f32 block scales: quantized in the prologue (fused) or copied from the
//     separate quantizer's output after griddepcontrol.wait (PDL);
//   - per 32-wide K block: ldmatrix A (16 rows x 32 B) and B (8 tokens x 32 B),
//     one m16n8k32 e4m3 MMA per 8 tokens from zero, then acc += d * sw * sx in
//     f32 (the block scales differ per block, so they are applied to each
//     block's exact-product partial);
//   - the S CTAs of a cluster hold the S K slices of one row tile; partials are
//     summed in fixed rank order through DSMEM, bias added, bf16 stored.
// Split-K depends on (N, K) only, so results do not depend on M.

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 16;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 64
constexpr int kStepBytes = 128;                     // K bytes per pipeline step
constexpr int kBoxBytes = kRowsPerWarp * kStepBytes;  // 2 KB TMA box
constexpr int kStages = 4;
constexpr int kRedPitch = kRowsPerCta + 4;  // floats per token row of the reduction tile

struct GemvParams {
  const uint8_t* codes;        // block [N/32, Kp/32] or row [N, Kp/32]
  const __nv_bfloat16* x;      // fused: [M, K]
  const uint8_t* xq;           // unfused: [M, Kp]
  const uint8_t* xcodes;       // unfused: [M, Kp/32]
  const __nv_bfloat16* bias;   // [N] or null
  __nv_bfloat16* out;          // [M, N]
  int M, N, K, Kp;
  int nsteps;                  // Kp / 128
  int splits;                  // cluster size along K
  int ks_max;                  // bytes of the largest K slice
};

struct SmemLayout {
  int wbuf, xbuf, sxf, wc, bars, total;
};

__host__ __device__ inline SmemLayout smem_layout(int ntok, int ks_max) {
  SmemLayout L;
  L.wbuf = 0;
  L.xbuf = kWarps * kStages * kBoxBytes;
  L.sxf = L.xbuf + ntok * ks_max;
  L.wc = L.sxf + ntok * (ks_max / 32) * 4;
  L.bars = ((L.wc + kRowsPerCta * (ks_max / 32)) + 15) & ~15;
  L.total = L.bars + kWarps * kStages * 8;
  return L;
}

// Byte offset of 16-byte chunk c of token t in the activation slice; chunks are
// XOR-swizzled by (t % 8) inside each 128-byte segment so ldmatrix over 8 tokens
// hits 8 different bank groups.
__device__ __forceinline__ int xchunk(int t, int c, int ks) {
  return t * ks + (((c & ~7) | ((c ^ t) & 7)) << 4);
}

template <int NT, bool kBlockScale, bool kFused>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const __grid_constant__ CUtensorMap wmap,
                                                           const GemvParams p) {
  constexpr int NTOK = NT * 8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // TMA 128B swizzle wants 1024-byte aligned boxes
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout L = smem_layout(NTOK, p.ks_max);
  uint8_t* wbuf = smem + L.wbuf;
  uint8_t* xbuf = smem + L.xbuf;
  float* sxf = reinterpret_cast<float*>(smem + L.sxf);
  uint8_t* wc = smem + L.wc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = (p.splits > 1) ? static_cast<int>(cluster_ctarank()) : 0;
  const int row0 = blockIdx.y * kRowsPerCta;
  const int base_steps = p.nsteps / p.splits, rem = p.nsteps % p.splits;
  const int st0 = split * base_steps + (split < rem ? split : rem);
  const int ns = base_steps + (split < rem ? 1 : 0);
  const int ks = ns * kStepBytes;   // this slice's bytes
  const int ksb = ks >> 5;          // this slice's MX blocks
  const int wrow0 = row0 + warp * kRowsPerWarp;

  pdl_launch_dependents();  // the next kernel may start streaming its own weights
  // ---- 1. start streaming this warp's weight rows (independent of earlier kernels)
  uint64_t* wbar = bars + warp * kStages;
  uint8_t* wst = wbuf + warp * kStages * kBoxBytes;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&wbar[s], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    const uint64_t pol = policy_evict_first();
    const int first = ns < kStages ? ns : kStages;
    for (int s = 0; s < first; ++s) {
      mbar_arrive_expect_tx(&wbar[s], kBoxBytes);
      tma_load_2d(wst + s * kBoxBytes, &wmap, &wbar[s], (st0 + s) * kStepBytes, wrow0, pol);
    }
  }

  // ---- 2. weight codes of the slice -> shared (immutable, read before any PDL wait)
  const int KBp = p.Kp >> 5;
  if (kBlockScale) {
    for (int i = threadIdx.x; i < 2 * ksb; i += blockDim.x) {
      const int g = i / ksb, j = i % ksb;
      const int grow = (row0 >> 5) + g;
      wc[g * ksb + j] = grow < (p.N >> 5) ? p.codes[static_cast<long long>(grow) * KBp + st0 * 4 + j] : 127;
    }
  } else {
    for (int i = threadIdx.x; i < kRowsPerCta * ksb; i += blockDim.x) {
      const int r = i / ksb, j = i % ksb;
      const int n = row0 + r;
      wc[r * ksb + j] = n < p.N ? p.codes[static_cast<long long>(n) * KBp + st0 * 4 + j] : 127;
    }
  }

  // ---- 3. activation slice -> shared (e4m3 bytes, swizzled) + f32 block scales
  const int k0 = st0 * kStepBytes;
  pdl_wait_prior_grid();  // x (and the quantizer's output) complete and visible
  if (kFused) {
    // quantize x[0..M) x [k0, k0 + ks) here: 8 elements a lane, 4 lanes a block
    const int gpr = ks >> 3;               // 8-element groups per token
    const int units = NTOK * gpr;          // multiple of 4
    for (int base = warp * 32; base < units; base += kWarps * 32) {
      const int u = base + lane;
      const bool inside = u < units;
      const int t = inside ? u / gpr : 0;
      const int q8 = inside ? u % gpr : 0;
      const int k = k0 + q8 * 8;
      const bool valid = inside && t < p.M && k < p.K;
      const uint4 xu = valid ? *reinterpret_cast<const uint4*>(p.x + static_cast<long long>(t) * p.K + k)
                             : make_uint4(0u, 0u, 0u, 0u);
      const QuantBlock8 b = mx_quant_bf16x8(xu);
      if (inside) {
        const uint2 qv = valid ? make_uint2(b.lo, b.hi) : make_uint2(0u, 0u);
        *reinterpret_cast<uint2*>(xbuf + xchunk(t, q8 >> 1, ks) + (q8 & 1) * 8) = qv;
        if ((q8 & 3) == 0) sxf[t * ksb + (q8 >> 2)] = valid ? e8m0_to_f32(b.code) : 0.0f;
      }
    }
  } else {
    const int cpr = ks >> 4;  // 16-byte chunks per token
    for (int i = threadIdx.x; i < NTOK * cpr; i += blockDim.x) {
      const int t = i / cpr, c = i % cpr;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t < p.M) v = *reinterpret_cast<const uint4*>(p.xq + static_cast<long long>(t) * p.Kp + k0 + c * 16);
      *reinterpret_cast<uint4*>(xbuf + xchunk(t, c, ks)) = v;
    }
    for (int i = threadIdx.x; i < NTOK * ksb; i += blockDim.x) {
      const int t = i / ksb, j = i % ksb;
      sxf[i] = t < p.M ? e8m0_to_f32(p.xcodes[static_cast<long long>(t) * KBp + st0 * 4 + j]) : 0.0f;
    }
  }
  __syncthreads();

  // ---- 4. main loop: this warp's 16 rows over the slice
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

  const int g = lane >> 2, tq = lane & 3;
  // ldmatrix row / chunk roles of this lane
  const int mi = lane >> 3;
  const int a_row = (lane & 7) + ((mi & 1) << 3);  // A: matrices (r0-7,c0) (r8-15,c0) (r0-7,c1) (r8-15,c1)
  const int a_chalf = mi >> 1;
  const int b_tok = (lane & 7) + ((mi >> 1) << 3);  // B x4: (t0-7,c0) (t0-7,c1) (t8-15,c0) (t8-15,c1)
  const int b_chalf = mi & 1;
  const uint32_t xbase = smem_u32(xbuf);
  const uint64_t pol = policy_evict_first();
  bool ok = true;

  for (int i = 0; i < ns; ++i) {
    const int slot = i % kStages;
    if (ok) ok = mbar_wait(&wbar[slot], (i / kStages) & 1);
    const uint32_t abase = smem_u32(wst + slot * kBoxBytes);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = i * 4 + j;  // MX block within the slice
      uint32_t a[4];
      {
        const int chunk = 2 * j + a_chalf;
        ldsm_x4(abase + a_row * kStepBytes + ((chunk ^ (a_row & 7)) << 4), a[0], a[1], a[2], a[3]);
      }
      float sw0, sw1;
      if (kBlockScale) {
        sw0 = sw1 = e8m0_to_f32(wc[(warp >> 1) * ksb + kb]);
      } else {
        sw0 = e8m0_to_f32(wc[(warp * kRowsPerWarp + g) * ksb + kb]);
        sw1 = e8m0_to_f32(wc[(warp * kRowsPerWarp + g + 8) * ksb + kb]);
      }
#pragma unroll
      for (int np = 0; np < (NT + 1) / 2; ++np) {
        uint32_t b[4];
        const int c = i * 8 + 2 * j + b_chalf;
        if (NT == 1) {
          const int t = lane & 7;
          ldsm_x2(xbase + xchunk(t, i * 8 + 2 * j + ((lane >> 3) & 1), ks), b[0], b[1]);
          b[2] = b[3] = 0u;
        } else {
          ldsm_x4(xbase + xchunk(np * 16 + b_tok, c, ks), b[0], b[1], b[2], b[3]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int nt = np * 2 + h;
          if (nt < NT) {
            float d[4];
            mma_e4m3_16832(d, a, b[2 * h], b[2 * h + 1]);
            const int t0 = nt * 8 + 2 * tq;
            const float sx0 = sxf[t0 * ksb + kb], sx1 = sxf[(t0 + 1) * ksb + kb];
            acc[nt][0] = fmaf(d[0], sw0 * sx0, acc[nt][0]);
            acc[nt][1] = fmaf(d[1], sw0 * sx1, acc[nt][1]);
            acc[nt][2] = fmaf(d[2], sw1 * sx0, acc[nt][2]);
            acc[nt][3] = fmaf(d[3], sw1 * sx1, acc[nt][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + kStages < ns && ok) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&wbar[slot], kBoxBytes);
      tma_load_2d(wst + slot * kBoxBytes, &wmap, &wbar[slot], (st0 + i + kStages) * kStepBytes, wrow0,
                  pol);
    }
  }
  __syncthreads();  // every TMA landed and every warp is done with its ring

  // ---- 5. partial tile [token][row] in shared memory (reuses the weight rings)
  float* red = reinterpret_cast<float*>(wbuf);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int t0 = nt * 8 + 2 * tq;
    const int r = warp * kRowsPerWarp + g;
    red[t0 * kRedPitch + r] = acc[nt][0];
    red[(t0 + 1) * kRedPitch + r] = acc[nt][1];
    red[t0 * kRedPitch + r + 8] = acc[nt][2];
    red[(t0 + 1) * kRedPitch + r + 8] = acc[nt][3];
  }

  // ---- 6. fixed-order split-K reduction across the cluster, bias, bf16 store
  const int S = p.splits;
  const int rows_per = kRowsPerCta / S;  // S divides 64
  const int r_begin = split * rows_per;
  if (S > 1) cluster_sync(); else __syncthreads();
  const uint32_t red_addr = smem_u32(red);
  const int Mv = p.M < NTOK ? p.M : NTOK;
  for (int idx = threadIdx.x; idx < Mv * rows_per; idx += blockDim.x) {
    const int t = idx / rows_per;
    const int r = r_begin + idx % rows_per;
    const int n = row0 + r;
    if (n >= p.N) continue;
    const uint32_t off = static_cast<uint32_t>((t * kRedPitch + r) * 4);
    float v = 0.0f;
    if (S > 1) {
      float part[8];
#pragma unroll
      for (int s = 0; s < 8; ++s)  // issue every rank's load before summing
        part[s] = s < S ? ld_shared_cluster_f32(map_shared_rank(red_addr + off, s)) : 0.0f;
#pragma unroll
      for (int s = 0; s < 8; ++s) v += part[s];  // fixed rank order
    } else {
      v = red[t * kRedPitch + r];
    }
    if (p.bias) v += __bfloat162float(p.bias[n]);
    p.out[static_cast<long long>(t) * p.N + n] = __float2bfloat16_rn(v);
  }
  if (S > 1) cluster_sync();  // peers may still be reading this CTA's partials
}

template <int NT, bool B, bool F>
int launch_one(const CUtensorMap& map, const GemvParams& p, int smem, bool pdl, cudaStream_t stream) {
  auto kern = gemv_kernel<NT, B, F>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "gemv: smem attribute: %s", cudaGetErrorString(e));
  if (p.splits > 1) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    (void)e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, (p.N + kRowsPerCta - 1) / kRowsPerCta, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = p.splits;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  (void)pdl;  // always a programmatic dependent: it waits before reading x
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, map, p);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "gemv launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

template <bool B, bool F>
int launch_nt(int nt, const CUtensorMap& map, const GemvParams& p, int smem, bool pdl, cudaStream_t s) {
  if (nt == 1) return launch_one<1, B, F>(map, p, smem, pdl, s);
  if (nt == 2) return launch_one<2, B, F>(map, p, smem, pdl, s);
  return launch_one<4, B, F>(map, p, smem, pdl, s);
}

}  // namespace

// Split count: enough CTAs for ~3 per SM, dividing the 64-row tile (1, 2, 4, 8),
// bounded by the K steps and by the activation slice that must fit in shared
// memory.  Depends on (N, Kp) and the token tile only, never on the values.
int gemv_splits(int N, int Kp, int M, int force_splits) {
  const int nsteps = Kp / kStepBytes;
  int S;
  if (force_splits > 0) {
    S = force_splits;
  } else {
    // smallest split giving ~2.5 CTAs per SM, so the whole grid is resident in
    // one wave and every warp's TMA boxes are in flight from the start
    DeviceInfo di;
    const int sms = current_device_info(&di) == MX_OK ? di.sm_count : 148;
    const int tiles = (N + kRowsPerCta - 1) / kRowsPerCta;
    S = 1;
    while (S < 8 && 2 * tiles * S < 5 * sms) S *= 2;
  }
  const int ntok = MX_GEMV_MAX_M;
  while (S < 8 && ntok * ((nsteps + S - 1) / S) * kStepBytes > 96 * 1024) S *= 2;
  while (S > 1 && S > nsteps) S >>= 1;
  return S;
}

unsigned int take_error_flags_gemv() { return take_tu_error_flags(); }

int launch_gemv(const GemvArgs& a, cudaStream_t stream) {
  const mx_packed_weight* w = a.w;
  GemvParams p = {};
  p.codes = w->codes;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.xq = a.xq;
  p.xcodes = a.xcodes;
  p.bias = static_cast<const __nv_bfloat16*>(a.bias);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = a.M;
  p.N = w->N;
  p.K = w->K;
  p.Kp = w->Kp;
  p.nsteps = w->Kp / kStepBytes;
  p.splits = gemv_splits(w->N, w->Kp, a.M, a.force_splits);
  if (kRowsPerCta % p.splits != 0 || p.splits > 8)
    return set_error(MX_ERR_ARG, "gemv: split count %d must be 1, 2, 4 or 8", p.splits);
  p.ks_max = ((p.nsteps + p.splits - 1) / p.splits) * kStepBytes;
  const int nt = a.M <= 8 ? 1 : (a.M <= 16 ? 2 : 4);
  const SmemLayout L = smem_layout(nt * 8, p.ks_max);
  const int smem = L.total + 1024;  // + alignment slack
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  if (static_cast<size_t>(smem) > di.max_smem_optin)
    return set_error(MX_ERR_UNSUPPORTED, "gemv: K = %d needs %d bytes of shared memory", w->K, smem);

  CUtensorMap map;
  int rc = encode_tensor_map_2d(&map, w->bytes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->Kp, w->N, w->Kp,
                                kStepBytes, kRowsPerWarp, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != MX_OK) return rc;
  const bool blk = w->scale_mode == MX_SCALE_BLOCK32X32;
  if (blk && a.fused) return launch_nt<true, true>(nt, map, p, smem, a.pdl, stream);
  if (blk && !a.fused) return launch_nt<true, false>(nt, map, p, smem, a.pdl, stream);
  if (!blk && a.fused) return launch_nt<false, true>(nt, map, p, smem, a.pdl, stream);
  return launch_nt<false, false>(nt, map, p, smem, a.pdl, stream);
}

}  // namespace mx
