// K-ROUTE (token -> expert grouping) and K-MOE (routed A16W4 expert GEMM).
//
// A16W4 product (a16w4 = vllm.models.minimax_m3.amd.specialized_decode.mono.a16w4,
// module text, dequant, step_mfma): MXFP4 weights are dequantized to bf16 in
// registers and multiplied by the bf16 token activations on tensor cores with
// f32 accumulation.  Here every e2m1 nibble becomes its exact bf16 value, one
// m16n8k16 bf16 MMA pair covers a 32-wide K block from zero, and the block's
// E8M0 factor 2^(c - 127) multiplies that f32 partial (exact up to f32 rounding
// of the product; the pages fold the factor into the bf16 operand instead).
//
// The packed weight stores, per 64-byte chunk of a row, word w of K block b at
// word 4 w + b, and inside each word the element pair (2i, 2i+1) at nibble slots
// (i, i + 4).  Lane (g, t) of a warp then reads its rows' four words for four K
// blocks with one 16-byte load (the "16 bytes a lane" lesson of weights942,
// fp4_lane_major / fp4_tile_major), and each bf16 pair is
//   ((w >> 4i) & 0x000F000F) * (2^6 + 2^12) & 0x81C081C0   (sign -> bit 15,
// exponent/mantissa -> bits 6..8, i.e. the value times 2^-126), times 2^126.
//
// Routing is the plainest reading of "routed experts" (the pages show no
// router): pairs grouped by expert id, stable in (token, slot) order.

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ pairs,
                 int32_t* __restrict__ active, int32_t* __restrict__ n_active, int* dev_status) {
  extern __shared__ int rs[];
  int* cnt = rs;           // [E]
  int* base = rs + E;      // [E]
  int* wcnt = rs + 2 * E;  // [warps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  int bad = 0;
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // integer counts: order-independent
    else if (e != -1) bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (warp == 0) {  // exclusive scan of the counts, and the ascending list of active experts
    int run = 0, arun = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? cnt[e] : 0;
      int incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned am = __ballot_sync(full, c > 0);
      if (e < E) {
        counts[e] = c;
        offsets[e] = run + incl - c;
        base[e] = run + incl - c;
        if (c > 0) active[arun + __popc(am & ((1u << lane) - 1u))] = e;
      }
      run += __shfl_sync(full, incl, 31);
      arun += __popc(am);
    }
    if (lane == 0) {
      offsets[E] = run;
      *n_active = arun;
      if (dev_status) *dev_status = bad ? MX_ERR_EXPERT_ID : MX_OK;
    }
  }
  __syncthreads();
  // stable scatter, blockDim pairs at a time: rank inside the warp by __match_any,
  // then the counts of the earlier warps, then the running base of the expert
  for (int c0 = 0; c0 < P; c0 += blockDim.x) {
    const int p = c0 + tid;
    const int e = p < P ? ids[p] : -1;
    const bool valid = e >= 0 && e < E;
    for (int i = lane; i < E; i += 32) wcnt[warp * E + i] = 0;
    __syncwarp();
    const unsigned key = valid ? static_cast<unsigned>(e) : static_cast<unsigned>(E + lane);
    const unsigned mask = __match_any_sync(full, key);
    const int rank = __popc(mask & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[warp * E + e] = __popc(mask);
    __syncthreads();
    if (valid) {
      int pos = base[e] + rank;
      for (int w = 0; w < warp; ++w) pos += wcnt[w * E + e];
      pairs[pos] = p;
    }
    __syncthreads();
    for (int i = tid; i < E; i += blockDim.x) {
      int s = 0;
      for (int w = 0; w < kRouteWarps; ++w) s += wcnt[w * E + i];
      base[i] += s;
    }
    __syncthreads();
  }
}

// One warp per pair: rows of pairs whose id is not a valid expert are zero.
__global__ void zero_invalid_pairs_kernel(const int32_t* __restrict__ ids, int P, int E, int N,
                                          __nv_bfloat16* __restrict__ out) {
  const int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (p >= P) return;
  const int e = ids[p];
  if (e >= 0 && e < E) return;
  const __nv_bfloat16 z = __float2bfloat16_rn(0.0f);
  for (int n = threadIdx.x & 31; n < N; n += 32) out[static_cast<long long>(p) * N + n] = z;
}

constexpr int kMoeWarps = 8;
constexpr int kMoeRows = kMoeWarps * 16;  // 128 weight rows a CTA
constexpr int kMoeTok = 16;               // tokens a chunk (two n8 tiles)
constexpr int kMoeStepK = 128;            // K elements a step (64 bytes a row)
constexpr int kPF = 4;                    // steps of weight words in flight a lane
constexpr int kMoeRedPitch = kMoeRows + 4;

struct MoeParams {
  const __nv_bfloat16* x;  // [T, K]
  const uint8_t* wq;       // [E, N, Kp/2]
  const uint8_t* codes;    // [E, N, Kp/32]
  const int32_t* offsets;
  const int32_t* pairs;
  const int32_t* active;
  const int32_t* n_active;
  __nv_bfloat16* out;      // [T * topk, N]
  int topk, N, K, Kp, nsteps, splits, ks_max;
};

// e2m1 x 8 (nibble slots (i, i+4) = elements (2i, 2i+1)) -> 4 bf16 pairs, exact.
MX_DEV void e2m1x8_to_bf16x8(uint32_t w, uint32_t (&r)[4]) {
  const __nv_bfloat162 two126 = __halves2bfloat162(__ushort_as_bfloat16(0x7e80),
                                                   __ushort_as_bfloat16(0x7e80));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = (w >> (4 * i)) & 0x000f000fu;
    const uint32_t v = (u * 0x1040u) & 0x81c081c0u;
    const __nv_bfloat162 b = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&v), two126);
    r[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// 16-byte chunk c of token row tk in the activation slice; the XOR by (tk & 1) * 4
// keeps the 8 lanes of a quarter warp (2 tokens x 4 chunks) on distinct banks.
MX_DEV int xs_chunk(int tk, int c) { return c ^ ((tk & 1) << 2); }

__global__ void __launch_bounds__(kMoeWarps * 32) moe_kernel(const MoeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* xs = smem;  // [kMoeTok][ks_max] bf16
  float* red = reinterpret_cast<float*>(smem + kMoeTok * p.ks_max * 2);
  int* tok_pair = reinterpret_cast<int*>(red + kMoeTok * kMoeRedPitch);

  const int a = blockIdx.z;
  if (a >= *p.n_active) return;  // same for every CTA of the cluster
  const int e = p.active[a];
  const int o0 = p.offsets[e];
  const int cnt = p.offsets[e + 1] - o0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int split = p.splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int base_steps = p.nsteps / p.splits, rem = p.nsteps % p.splits;
  const int st0 = split * base_steps + (split < rem ? split : rem);
  const int ns = base_steps + (split < rem ? 1 : 0);
  const int ks = ns * kMoeStepK;      // slice K elements
  const int kxb = ks * 2;             // slice bytes of one token row
  const int row0 = blockIdx.y * kMoeRows;
  const int rg = row0 + warp * 16 + g;  // rows rg and rg + 8
  const int KHp = p.Kp >> 1, KBp = p.Kp >> 5;
  const bool v0 = rg < p.N, v1 = rg + 8 < p.N;
  const long long erow = static_cast<long long>(e) * p.N;
  const uint8_t* w0 = p.wq + (erow + (v0 ? rg : 0)) * KHp + st0 * 64 + tq * 16;
  const uint8_t* w1 = p.wq + (erow + (v1 ? rg + 8 : 0)) * KHp + st0 * 64 + tq * 16;
  const uint8_t* c0p = p.codes + (erow + (v0 ? rg : 0)) * KBp + st0 * 4;
  const uint8_t* c1p = p.codes + (erow + (v1 ? rg + 8 : 0)) * KBp + st0 * 4;
  const uint32_t xs_base = smem_u32(xs);

  for (int ch = 0; ch < cnt; ch += kMoeTok) {
    // ---- stage the chunk's token rows of the K slice (bf16, swizzled 16-byte chunks)
    if (threadIdx.x < kMoeTok)
      tok_pair[threadIdx.x] = (ch + static_cast<int>(threadIdx.x) < cnt) ? p.pairs[o0 + ch + threadIdx.x] : -1;
    __syncthreads();
    const int cpt = ks >> 3;  // 16-byte chunks a token row
    for (int i = threadIdx.x; i < kMoeTok * cpt; i += blockDim.x) {
      const int tk = i / cpt, c = i % cpt;
      const int pr = tok_pair[tk];
      const int k = st0 * kMoeStepK + c * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (pr >= 0 && k < p.K)
        v = *reinterpret_cast<const uint4*>(p.x + static_cast<long long>(pr / p.topk) * p.K + k);
      *reinterpret_cast<uint4*>(xs + tk * kxb + xs_chunk(tk, c) * 16) = v;
    }
    __syncthreads();

    // ---- K loop: 16 rows a warp, two n8 token tiles
    float acc[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = 0.0f;
    uint4 wb0[kPF], wb1[kPF];
    uint32_t cb0[kPF], cb1[kPF];
#pragma unroll
    for (int q = 0; q < kPF; ++q) {
      if (q < ns) {
        wb0[q] = v0 ? ld_nc_v4(w0 + q * 64) : make_uint4(0u, 0u, 0u, 0u);
        wb1[q] = v1 ? ld_nc_v4(w1 + q * 64) : make_uint4(0u, 0u, 0u, 0u);
        cb0[q] = *reinterpret_cast<const uint32_t*>(c0p + q * 4);
        cb1[q] = *reinterpret_cast<const uint32_t*>(c1p + q * 4);
      }
    }
    for (int i0 = 0; i0 < ns; i0 += kPF) {
#pragma unroll
      for (int q = 0; q < kPF; ++q) {
        const int i = i0 + q;
        if (i < ns) {
          const uint32_t wa[4] = {wb0[q].x, wb0[q].y, wb0[q].z, wb0[q].w};
          const uint32_t wc[4] = {wb1[q].x, wb1[q].y, wb1[q].z, wb1[q].w};
          const uint32_t ca = cb0[q], cc = cb1[q];
          if (i + kPF < ns) {  // refill this slot with step i + kPF
            wb0[q] = v0 ? ld_nc_v4(w0 + (i + kPF) * 64) : make_uint4(0u, 0u, 0u, 0u);
            wb1[q] = v1 ? ld_nc_v4(w1 + (i + kPF) * 64) : make_uint4(0u, 0u, 0u, 0u);
            cb0[q] = *reinterpret_cast<const uint32_t*>(c0p + (i + kPF) * 4);
            cb1[q] = *reinterpret_cast<const uint32_t*>(c1p + (i + kPF) * 4);
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t ra[4], rc[4];
            e2m1x8_to_bf16x8(wa[b], ra);
            e2m1x8_to_bf16x8(wc[b], rc);
            const float s0 = e8m0_to_f32((ca >> (8 * b)) & 0xffu);
            const float s1 = e8m0_to_f32((cc >> (8 * b)) & 0xffu);
            const int c = i * 16 + b * 4 + tq;  // 16-byte chunk: logical k = 8c .. 8c + 7
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int tk = h * 8 + g;
              uint4 xv;
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                           : "r"(xs_base + tk * kxb + xs_chunk(tk, c) * 16));
              float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
              mma_bf16_16816(d, ra[0], rc[0], ra[1], rc[1], xv.x, xv.y);
              mma_bf16_16816(d, ra[2], rc[2], ra[3], rc[3], xv.z, xv.w);
              acc[h][0] = fmaf(d[0], s0, acc[h][0]);
              acc[h][1] = fmaf(d[1], s0, acc[h][1]);
              acc[h][2] = fmaf(d[2], s1, acc[h][2]);
              acc[h][3] = fmaf(d[3], s1, acc[h][3]);
            }
          }
        }
      }
    }

    // ---- partial tile [token][row], fixed-order cluster reduction, bf16 store
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t0 = h * 8 + 2 * tq;
      const int r = warp * 16 + g;
      red[t0 * kMoeRedPitch + r] = acc[h][0];
      red[(t0 + 1) * kMoeRedPitch + r] = acc[h][1];
      red[t0 * kMoeRedPitch + r + 8] = acc[h][2];
      red[(t0 + 1) * kMoeRedPitch + r + 8] = acc[h][3];
    }
    const int S = p.splits;
    if (S > 1) cluster_sync(); else __syncthreads();
    const int rows_per = kMoeRows / S;
    const int r_begin = split * rows_per;
    const int nt = (cnt - ch) < kMoeTok ? (cnt - ch) : kMoeTok;
    const uint32_t red_addr = smem_u32(red);
    for (int idx = threadIdx.x; idx < nt * rows_per; idx += blockDim.x) {
      const int t = idx / rows_per;
      const int r = r_begin + idx % rows_per;
      const int n = row0 + r;
      if (n >= p.N) continue;
      const uint32_t off = static_cast<uint32_t>((t * kMoeRedPitch + r) * 4);
      float v = 0.0f;
      if (S > 1) {
        for (int s = 0; s < S; ++s) v += ld_shared_cluster_f32(map_shared_rank(red_addr + off, s));
      } else {
        v = red[t * kMoeRedPitch + r];
      }
      p.out[static_cast<long long>(tok_pair[t]) * p.N + n] = __float2bfloat16_rn(v);
    }
    if (S > 1) cluster_sync(); else __syncthreads();
  }
}

int moe_splits(int Kp, int N, int zmax, int sms) {
  const int nsteps = Kp / kMoeStepK;
  int S = 1;
  while (S < 8 && ((nsteps + S - 1) / S) * kMoeStepK * 2 * kMoeTok > 64 * 1024) S *= 2;
  const long long tiles = static_cast<long long>((N + kMoeRows - 1) / kMoeRows) * zmax;
  while (S < 8 && tiles * S < 2LL * sms && (nsteps + 2 * S - 1) / (2 * S) >= kPF) S *= 2;
  while (S > 1 && S > nsteps) S >>= 1;
  return S;
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, int T, int topk, int E, int32_t* counts,
                         int32_t* offsets, int32_t* pairs, int32_t* active, int32_t* n_active,
                         int* dev_status, cudaStream_t stream) {
  const int smem = (2 * E + kRouteWarps * E) * static_cast<int>(sizeof(int));
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  route_kernel<<<1, kRouteThreads, smem, stream>>>(ids, T * topk, E, counts, offsets, pairs, active,
                                                   n_active, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_zero_invalid_pairs(const int32_t* ids, int T, int topk, int E, int N, void* out,
                                      cudaStream_t stream) {
  const int P = T * topk;
  const int warps = 8;
  zero_invalid_pairs_kernel<<<(P + warps - 1) / warps, warps * 32, 0, stream>>>(
      ids, P, E, N, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

int launch_moe(const void* x, int T, int topk, const mx_packed_weight* w, const int32_t* offsets,
               const int32_t* pairs, const int32_t* active, const int32_t* n_active, void* out,
               cudaStream_t stream) {
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  MoeParams p = {};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.wq = w->bytes;
  p.codes = w->codes;
  p.offsets = offsets;
  p.pairs = pairs;
  p.active = active;
  p.n_active = n_active;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.topk = topk;
  p.N = w->N;
  p.K = w->K;
  p.Kp = w->Kp;
  p.nsteps = w->Kp / kMoeStepK;
  const long long P = static_cast<long long>(T) * topk;
  const int zmax = static_cast<int>(P < w->E ? P : w->E);
  p.splits = moe_splits(w->Kp, w->N, zmax, di.sm_count);
  p.ks_max = ((p.nsteps + p.splits - 1) / p.splits) * kMoeStepK;
  const int smem = kMoeTok * p.ks_max * 2 + kMoeTok * kMoeRedPitch * 4 + kMoeTok * 4;
  if (static_cast<size_t>(smem) > di.max_smem_optin)
    return set_error(MX_ERR_UNSUPPORTED, "moe: K = %d needs %d bytes of shared memory", w->K, smem);
  cudaError_t e = cudaFuncSetAttribute(moe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe: smem attribute: %s", cudaGetErrorString(e));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, (w->N + kMoeRows - 1) / kMoeRows, zmax);
  cfg.blockDim = dim3(kMoeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = p.splits;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, moe_kernel, p);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

}  // namespace mx
