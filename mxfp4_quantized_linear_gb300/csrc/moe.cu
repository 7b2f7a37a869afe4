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
constexpr int kChunkK = 256;              // K elements of activation a ring slot (2 steps)
constexpr int kChunkBytes = kMoeTok * kChunkK * 2;  // 8 KB
constexpr int kPF = 4;                    // steps of weight words in flight a lane

struct MoeParams {
  const __nv_bfloat16* x;  // [T, K]
  const uint8_t* wq;       // [E, N, Kp/2]
  const uint8_t* codes;    // [E, N, Kp/32]
  const int32_t* offsets;
  const int32_t* pairs;
  const int32_t* active;
  const int32_t* n_active;
  __nv_bfloat16* out;      // [T * topk, N]
  int topk, N, K, Kp, nsteps;
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

// 16-byte chunk c (0..31) of token row tk in an activation ring slot; the XOR by
// (tk & 1) * 4 keeps the 8 lanes of a quarter warp (2 tokens x 4 chunks) on
// distinct banks.
MX_DEV int xs_off(int tk, int c) { return tk * (kChunkK * 2) + ((c ^ ((tk & 1) << 2)) << 4); }

MX_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
MX_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MX_DEV void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// One step of one warp: 16 weight rows x 128 K against up to 16 tokens.
MX_DEV void moe_step(float (&acc)[2][4], const uint4& wa4, const uint4& wc4, uint32_t ca, uint32_t cc,
                     uint32_t xs_base, int s_in_chunk, int g, int tq) {
  const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
  const uint32_t wc[4] = {wc4.x, wc4.y, wc4.z, wc4.w};
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t ra[4], rc[4];
    e2m1x8_to_bf16x8(wa[b], ra);
    e2m1x8_to_bf16x8(wc[b], rc);
    const float s0 = e8m0_to_f32((ca >> (8 * b)) & 0xffu);
    const float s1 = e8m0_to_f32((cc >> (8 * b)) & 0xffu);
    const int c = s_in_chunk * 16 + b * 4 + tq;  // 16-byte chunk: K = 8c .. 8c + 7 of the slot
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tk = h * 8 + g;
      uint4 xv;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                   : "r"(xs_base + xs_off(tk, c)));
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

__global__ void __launch_bounds__(kMoeWarps * 32, 1) moe_kernel(const MoeParams p) {
  __shared__ __align__(128) uint8_t xs[2][kChunkBytes];
  __shared__ int tok_src[kMoeTok];   // token row of x, or -1
  __shared__ int tok_pair[kMoeTok];  // output row (pair index), or -1

  const int a = blockIdx.y;
  if (a >= *p.n_active) return;
  const int e = p.active[a];
  const int o0 = p.offsets[e];
  const int cnt = p.offsets[e + 1] - o0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int row0 = blockIdx.x * kMoeRows;
  const int rg = row0 + warp * 16 + g;  // rows rg and rg + 8
  const int KHp = p.Kp >> 1, KBp = p.Kp >> 5;
  const bool v0 = rg < p.N, v1 = rg + 8 < p.N;
  const long long erow = static_cast<long long>(e) * p.N;
  const uint8_t* w0 = p.wq + (erow + (v0 ? rg : 0)) * KHp + tq * 16;
  const uint8_t* w1 = p.wq + (erow + (v1 ? rg + 8 : 0)) * KHp + tq * 16;
  const uint8_t* c0p = p.codes + (erow + (v0 ? rg : 0)) * KBp;
  const uint8_t* c1p = p.codes + (erow + (v1 ? rg + 8 : 0)) * KBp;
  const int ns = p.nsteps;
  const int nchunks = (ns + 1) >> 1;

  for (int ch = 0; ch < cnt; ch += kMoeTok) {
    // ---- 1. weights of the first kPF steps: independent of the activations
    uint4 wb0[kPF], wb1[kPF];
    uint32_t cb0[kPF], cb1[kPF];
#pragma unroll
    for (int q = 0; q < kPF; ++q) {
      const bool in = q < ns;
      wb0[q] = (in && v0) ? ld_nc_v4(w0 + q * 64) : make_uint4(0u, 0u, 0u, 0u);
      wb1[q] = (in && v1) ? ld_nc_v4(w1 + q * 64) : make_uint4(0u, 0u, 0u, 0u);
      cb0[q] = in ? *reinterpret_cast<const uint32_t*>(c0p + q * 4) : 0x7f7f7f7fu;
      cb1[q] = in ? *reinterpret_cast<const uint32_t*>(c1p + q * 4) : 0x7f7f7f7fu;
    }
    // ---- 2. the chunk's tokens, and the first two activation slots
    if (threadIdx.x < kMoeTok) {
      const int pr = (ch + static_cast<int>(threadIdx.x) < cnt) ? p.pairs[o0 + ch + threadIdx.x] : -1;
      tok_pair[threadIdx.x] = pr;
      tok_src[threadIdx.x] = pr >= 0 ? pr / p.topk : -1;
    }
    __syncthreads();
    auto load_slot = [&](int c, int buf) {
      const uint32_t dst = smem_u32(xs[buf]);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int idx = threadIdx.x + j * kMoeWarps * 32;  // 512 chunks of 16 bytes
        const int tk = idx >> 5, cc = idx & 31;
        const int src = tok_src[tk];
        const int k = c * kChunkK + cc * 8;
        const bool ok = src >= 0 && k < p.K && c < nchunks;
        const __nv_bfloat16* sp = ok ? p.x + static_cast<long long>(src) * p.K + k : p.x;
        cp_async16(dst + xs_off(tk, cc), sp, ok);
      }
      cp_async_commit();
    };
    load_slot(0, 0);
    load_slot(1, 1);

    // ---- 3. K loop: two slots (four steps) an iteration so register slots stay static
    float acc[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = 0.0f;
    for (int c0 = 0; c0 < nchunks; c0 += 2) {
#pragma unroll
      for (int cs = 0; cs < 2; ++cs) {
        const int c = c0 + cs;
        if (c < nchunks) {
          cp_async_wait1();
          __syncthreads();
          const uint32_t xs_base = smem_u32(xs[cs]);
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const int q = cs * 2 + s;  // register slot (static)
            const int i = c * 2 + s;   // step
            if (i < ns) {
              const uint4 wa = wb0[q], wc = wb1[q];
              const uint32_t ca = cb0[q], cc = cb1[q];
              if (i + kPF < ns) {
                wb0[q] = v0 ? ld_nc_v4(w0 + (i + kPF) * 64) : make_uint4(0u, 0u, 0u, 0u);
                wb1[q] = v1 ? ld_nc_v4(w1 + (i + kPF) * 64) : make_uint4(0u, 0u, 0u, 0u);
                cb0[q] = *reinterpret_cast<const uint32_t*>(c0p + (i + kPF) * 4);
                cb1[q] = *reinterpret_cast<const uint32_t*>(c1p + (i + kPF) * 4);
              }
              moe_step(acc, wa, wc, ca, cc, xs_base, s, g, tq);
            }
          }
          __syncthreads();  // every warp is done with this slot
          load_slot(c + 2, cs);
        }
      }
    }

    // ---- 4. store: out[pair, row] (pairs with no token stay untouched)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t0 = h * 8 + 2 * tq;
      const int pa = tok_pair[t0], pb = tok_pair[t0 + 1];
      if (pa >= 0 && v0) p.out[static_cast<long long>(pa) * p.N + rg] = __float2bfloat16_rn(acc[h][0]);
      if (pb >= 0 && v0) p.out[static_cast<long long>(pb) * p.N + rg] = __float2bfloat16_rn(acc[h][1]);
      if (pa >= 0 && v1) p.out[static_cast<long long>(pa) * p.N + rg + 8] = __float2bfloat16_rn(acc[h][2]);
      if (pb >= 0 && v1) p.out[static_cast<long long>(pb) * p.N + rg + 8] = __float2bfloat16_rn(acc[h][3]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();  // tok_* and the ring are reused by the next chunk of tokens
  }
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
  dim3 grid((w->N + kMoeRows - 1) / kMoeRows, zmax, 1);
  moe_kernel<<<grid, kMoeWarps * 32, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

}  // namespace mx
