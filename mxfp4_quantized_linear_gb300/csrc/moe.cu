// K-ROUTE (token -> expert grouping) and K-MOE (routed A16W4 expert GEMM).
//
// A16W4 product (a16w4 = vllm.models.minimax_m3.amd.specialized_decode.mono.a16w4,
// module text, dequant, step_mfma): MXFP4 weights are dequantized to bf16 in
// registers and multiplied by the bf16 token activations on tensor cores with
// f32 accumulation.  Here, as on the page, every e2m1 nibble becomes the bf16
// value of the dequantized weight e2m1 x 2^(c - 127) (exact: a power-of-two
// multiply of an exact bf16), and the m16n8k16 bf16 MMAs accumulate the whole
// K extent straight into the f32 accumulators.
//
// The packed weight stores, per 64-byte chunk of a row, word w of K block b at
// word 4 w + b, and inside each word the element pair (2i, 2i+1) at nibble slots
// (i, i + 4).  Lane (g, t) of a warp then reads its rows' four words for four K
// blocks with one 16-byte load (the "16 bytes a lane" lesson of weights942,
// fp4_lane_major / fp4_tile_major), and each bf16 pair is
//   ((w >> 4i) & 0x000F000F) * (2^6 + 2^12) & 0x81C081C0   (sign -> bit 15,
// exponent/mantissa -> bits 6..8, i.e. the value times 2^-126), times 2^126,
// times the block's 2^(c - 127).
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

// out[t, h] = bf16(sum_j w[t, j] y2[t * topk + j, h]) over the slots j with a
// valid expert id, in increasing j, in f32: one thread per 4 consecutive h.
__global__ void combine_kernel(const float* __restrict__ y2, const int32_t* __restrict__ ids,
                               const float* __restrict__ wts, int T, int topk, int E, int H,
                               __nv_bfloat16* __restrict__ out) {
  const int H4 = H >> 2;
  const long long total = static_cast<long long>(T) * H4;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H4), h = static_cast<int>(i % H4) * 4;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j = 0; j < topk; ++j) {
      const int e = ids[t * topk + j];
      if (e < 0 || e >= E) continue;
      const float w = wts[t * topk + j];
      const float4 v = *reinterpret_cast<const float4*>(y2 + static_cast<long long>(t * topk + j) * H + h);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    *reinterpret_cast<uint2*>(out + static_cast<long long>(t) * H + h) =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

constexpr int kMoeOutBf16 = 0;    // out [pairs, N] bf16 (rows in gate-then-up order)
constexpr int kMoeOutSwiglu = 1;  // out [pairs, N/2] bf16 = silu(gate) * up
constexpr int kMoeOutF32 = 2;     // out_f32 [pairs, N] f32

constexpr int kMoeWarps = 8;
constexpr int kMoeRows = kMoeWarps * 16;  // 128 weight rows a CTA
constexpr int kMoeTok = 16;               // tokens a chunk (two n8 tiles)
constexpr int kStageSteps = 4;            // 128-wide K steps a ring stage (256 bytes a row)
constexpr int kStageK = kStageSteps * 128;                   // 512 K elements
constexpr int kWarpStageBytes = 16 * kStageSteps * 64;       // 4 KB: two 16x128-byte boxes
constexpr int kRing = 2;                                     // stages a warp keeps in flight
constexpr int kChunkBytes = kMoeTok * kStageK * 2;           // 16 KB of bf16 activations a stage
constexpr int kMoeSmem = kMoeWarps * kRing * kWarpStageBytes + 2 * kChunkBytes + 1024;

struct MoeParams {
  const __nv_bfloat16* x;  // [T, K] (one row a token) or [T * topk, K] (one row a pair)
  const uint8_t* codes;    // [E, N, Kp/32]
  const int32_t* offsets;
  const int32_t* pairs;
  const int32_t* active;
  const int32_t* n_active;
  __nv_bfloat16* out;      // kMoeOutBf16: [T * topk, N]; kMoeOutSwiglu: [T * topk, N / 2]
  float* out_f32;          // kMoeOutF32: [T * topk, N]
  int topk, N, K, Kp, nsteps;
  int x_per_pair;          // 1: activation row = pair index (the down projection)
  int gate_up;             // weight rows interleaved gate / up in 8-row groups
  int out_mode;
};

// E8M0 code c of one block -> bf16x2 {2^(c-127), 2^(c-127)}: exponent field c
// in both halves; code 0 -> the bf16 subnormal 2^-127 (0x0040).  Weight codes
// are never 255 (the packer rejects them).
MX_DEV uint32_t e8m0_to_bf16x2(uint32_t c) { return __vmaxu2(c * 0x00800080u, 0x00400040u); }

// e2m1 x 8 (nibble slots (i, i+4) = elements (2i, 2i+1)) -> 4 bf16 pairs of the
// dequantized weight e2m1 x 2^(c-127), exact (a16w4, dequant: fp4 with its
// E8M0 scale to bf16).  The sign and the 3 exponent/mantissa bits land in a
// bf16 whose value is the e2m1 value x 2^-126 (e2m1 subnormals map onto bf16
// subnormals); two power-of-two multiplies give the scaled value.
MX_DEV void e2m1x8_to_bf16x8_scaled(uint32_t w, uint32_t scale2, uint32_t (&r)[4]) {
  const __nv_bfloat162 two126 = __halves2bfloat162(__ushort_as_bfloat16(0x7e80),
                                                   __ushort_as_bfloat16(0x7e80));
  const __nv_bfloat162 sc = *reinterpret_cast<const __nv_bfloat162*>(&scale2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = (w >> (4 * i)) & 0x000f000fu;
    const uint32_t v = (u * 0x1040u) & 0x81c081c0u;
    const __nv_bfloat162 b = __hmul2(__hmul2(*reinterpret_cast<const __nv_bfloat162*>(&v), two126), sc);
    r[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// 16-byte chunk c (0..63) of token row tk in an activation stage; the XOR by
// (tk & 1) * 4 keeps the 8 lanes of a quarter warp (2 tokens x 4 chunks) on
// distinct banks.
MX_DEV int xs_off(int tk, int c) { return tk * (kStageK * 2) + ((c ^ ((tk & 1) << 2)) << 4); }

MX_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
MX_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MX_DEV void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

MX_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Packed row r of a gate / up interleaved weight -> its row in gate-then-up order.
MX_DEV int gate_up_row(int r, int N) {
  const int q = r >> 4, i = r & 15;
  return i < 8 ? 8 * q + i : (N >> 1) + 8 * q + i - 8;
}

MX_DEV float silu_f32(float v) { return v / (1.0f + expf(-v)); }

__global__ void __launch_bounds__(kMoeWarps * 32, 2) moe_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                const MoeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;                                              // [warp][kRing][4 KB]
  uint8_t* xs = smem + kMoeWarps * kRing * kWarpStageBytes;           // [2][16 KB]
  __shared__ uint64_t bars[kMoeWarps][kRing];
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
  const int wrow = row0 + warp * 16;        // this warp's first row within the expert
  const int rg = wrow + g;                   // rows rg and rg + 8
  const int KBp = p.Kp >> 5;
  const bool v0 = rg < p.N, v1 = rg + 8 < p.N;
  const long long erow = static_cast<long long>(e) * p.N;
  const uint8_t* c0p = p.codes + (erow + (v0 ? rg : 0)) * KBp;
  const uint8_t* c1p = p.codes + (erow + (v1 ? rg + 8 : 0)) * KBp;
  const int nst = (p.nsteps + kStageSteps - 1) / kStageSteps;  // ring stages along K
  uint8_t* myring = wring + warp * kRing * kWarpStageBytes;
  uint64_t* mybar = bars[warp];
  const int grow = static_cast<int>(erow) + wrow;               // row in the flattened [E*N] map
  const uint64_t pol = policy_evict_first();
  uint32_t uses = 0;  // parity of each ring slot's next completion

  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();
  auto issue = [&](int st, int slot) {  // weights of ring stage st (4 steps, 16 rows)
    uint8_t* dst = myring + slot * kWarpStageBytes;
    mbar_arrive_expect_tx(&mybar[slot], kWarpStageBytes);
    tma_load_2d(dst, &wmap, &mybar[slot], st * 256, grow, pol);
    tma_load_2d(dst + 2048, &wmap, &mybar[slot], st * 256 + 128, grow, pol);
  };

  for (int ch = 0; ch < cnt; ch += kMoeTok) {
    // ---- 1. weight stages 0..kRing-1 (independent of the tokens)
    if (lane == 0)
      for (int s = 0; s < kRing && s < nst; ++s) issue(s, s);
    // ---- 2. the chunk's tokens and the first two activation stages
    if (threadIdx.x < kMoeTok) {
      const int pr = (ch + static_cast<int>(threadIdx.x) < cnt) ? p.pairs[o0 + ch + threadIdx.x] : -1;
      tok_pair[threadIdx.x] = pr;
      tok_src[threadIdx.x] = pr >= 0 ? (p.x_per_pair ? pr : pr / p.topk) : -1;
    }
    __syncthreads();
    auto load_x = [&](int st, int buf) {
      const uint32_t dst = smem_u32(xs + buf * kChunkBytes);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = threadIdx.x + j * kMoeWarps * 32;  // 1024 chunks of 16 bytes
        const int tk = idx >> 6, cc = idx & 63;
        const int src = tok_src[tk];
        const int k = st * kStageK + cc * 8;
        const bool ok = src >= 0 && k < p.K && st < nst;
        const __nv_bfloat16* sp = ok ? p.x + static_cast<long long>(src) * p.K + k : p.x;
        cp_async16(dst + xs_off(tk, cc), sp, ok);
      }
      cp_async_commit();
    };
    load_x(0, 0);
    load_x(1, 1);
    uint4 cnext0, cnext1;  // codes of the next stage: 4 steps x 4 blocks, rows rg and rg + 8
    auto load_codes = [&](int st, uint4& c0, uint4& c1) {
      const uint32_t* a0 = reinterpret_cast<const uint32_t*>(c0p + st * 16);
      const uint32_t* a1 = reinterpret_cast<const uint32_t*>(c1p + st * 16);
      const int nsl = p.nsteps - st * kStageSteps;  // steps of this stage that exist
      c0.x = a0[0]; c1.x = a1[0];
      c0.y = nsl > 1 ? a0[1] : 0x7f7f7f7fu; c1.y = nsl > 1 ? a1[1] : 0x7f7f7f7fu;
      c0.z = nsl > 2 ? a0[2] : 0x7f7f7f7fu; c1.z = nsl > 2 ? a1[2] : 0x7f7f7f7fu;
      c0.w = nsl > 3 ? a0[3] : 0x7f7f7f7fu; c1.w = nsl > 3 ? a1[3] : 0x7f7f7f7fu;
    };
    load_codes(0, cnext0, cnext1);
    // a chunk of at most 8 tokens needs only the first n8 tile of the MMA
    const int ntile = (cnt - ch) > 8 ? 2 : 1;

    float acc[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = 0.0f;

    for (int st = 0; st < nst; ++st) {
      const int slot = st % kRing;
      const uint4 cs0 = cnext0, cs1 = cnext1;
      if (st + 1 < nst) load_codes(st + 1, cnext0, cnext1);
      cp_async_wait1();
      __syncthreads();  // activation stage st is in shared memory for every warp
      mbar_wait(&mybar[slot], (uses >> slot) & 1u);
      const uint32_t wbase = smem_u32(myring + slot * kWarpStageBytes);
      const uint32_t xbase = smem_u32(xs + (st & 1) * kChunkBytes);
      const uint32_t c0w[4] = {cs0.x, cs0.y, cs0.z, cs0.w};
      const uint32_t c1w[4] = {cs1.x, cs1.y, cs1.z, cs1.w};
#pragma unroll
      for (int s = 0; s < kStageSteps; ++s) {
        if (st * kStageSteps + s < p.nsteps) {
          // this lane's 16 bytes (4 K blocks, word tq) of rows g and g + 8; box s / 2,
          // 128B swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
          const int c = (s & 1) * 4 + tq;
          const uint32_t box = wbase + (s >> 1) * 2048;
          const uint4 wa4 = ld_shared_v4(box + g * 128 + ((c ^ g) << 4));
          const uint4 wc4 = ld_shared_v4(box + (g + 8) * 128 + ((c ^ g) << 4));
          const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
          const uint32_t wc[4] = {wc4.x, wc4.y, wc4.z, wc4.w};
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t ra[4], rc[4];
            e2m1x8_to_bf16x8_scaled(wa[b], e8m0_to_bf16x2((c0w[s] >> (8 * b)) & 0xffu), ra);
            e2m1x8_to_bf16x8_scaled(wc[b], e8m0_to_bf16x2((c1w[s] >> (8 * b)) & 0xffu), rc);
            const int xc = s * 16 + b * 4 + tq;  // 16-byte activation chunk: K = 8 xc .. + 7
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h >= ntile) break;  // block-uniform
              const int tk = h * 8 + g;
              const uint4 xv = ld_shared_v4(xbase + xs_off(tk, xc));
              // the weights carry their block scale: accumulate straight into acc
              mma_bf16_16816(acc[h], ra[0], rc[0], ra[1], rc[1], xv.x, xv.y);
              mma_bf16_16816(acc[h], ra[2], rc[2], ra[3], rc[3], xv.z, xv.w);
            }
          }
        }
      }
      uses ^= 1u << slot;
      __syncwarp();
      if (lane == 0 && st + kRing < nst) issue(st + kRing, slot);
      __syncthreads();  // every warp is done with activation stage st
      load_x(st + 2, st & 1);
    }

    // ---- 3. store the chunk's rows: acc[h][0..1] are row rg, [2..3] row rg + 8,
    // columns (tokens) h * 8 + 2 tq and + 1
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t0 = h * 8 + 2 * tq;
      const int pa = tok_pair[t0], pb = tok_pair[t0 + 1];
      if (p.out_mode == kMoeOutSwiglu) {
        // rows rg (gate) and rg + 8 (up) are gate / up of intermediate index i
        const int I = p.N >> 1, i = (wrow >> 1) + g;
        if (pa >= 0 && v1)
          p.out[static_cast<long long>(pa) * I + i] = __float2bfloat16_rn(silu_f32(acc[h][0]) * acc[h][2]);
        if (pb >= 0 && v1)
          p.out[static_cast<long long>(pb) * I + i] = __float2bfloat16_rn(silu_f32(acc[h][1]) * acc[h][3]);
      } else if (p.out_mode == kMoeOutF32) {
        if (pa >= 0 && v0) p.out_f32[static_cast<long long>(pa) * p.N + rg] = acc[h][0];
        if (pb >= 0 && v0) p.out_f32[static_cast<long long>(pb) * p.N + rg] = acc[h][1];
        if (pa >= 0 && v1) p.out_f32[static_cast<long long>(pa) * p.N + rg + 8] = acc[h][2];
        if (pb >= 0 && v1) p.out_f32[static_cast<long long>(pb) * p.N + rg + 8] = acc[h][3];
      } else {
        const int n0 = p.gate_up ? gate_up_row(rg, p.N) : rg;
        const int n1 = p.gate_up ? gate_up_row(rg + 8, p.N) : rg + 8;
        if (pa >= 0 && v0) p.out[static_cast<long long>(pa) * p.N + n0] = __float2bfloat16_rn(acc[h][0]);
        if (pb >= 0 && v0) p.out[static_cast<long long>(pb) * p.N + n0] = __float2bfloat16_rn(acc[h][1]);
        if (pa >= 0 && v1) p.out[static_cast<long long>(pa) * p.N + n1] = __float2bfloat16_rn(acc[h][2]);
        if (pb >= 0 && v1) p.out[static_cast<long long>(pb) * p.N + n1] = __float2bfloat16_rn(acc[h][3]);
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();  // tok_* and the buffers are reused by the next chunk of tokens
  }
}

}  // namespace

unsigned int take_error_flags_moe() { return take_tu_error_flags(); }

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

cudaError_t launch_combine(const float* y2, const int32_t* ids, const float* wts, int T, int topk, int E, int H,
                           void* out, cudaStream_t stream) {
  const long long total = static_cast<long long>(T) * (H / 4);
  combine_kernel<<<blocks_for(total, 256), 256, 0, stream>>>(y2, ids, wts, T, topk, E, H,
                                                             static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

int launch_moe(const MoeLaunch& a, cudaStream_t stream) {
  const mx_packed_weight* w = a.w;
  const void* x = a.x;
  const int T = a.T, topk = a.topk;
  MoeParams p = {};
  p.x_per_pair = a.x_per_pair;
  p.gate_up = w->layout == MX_LAYOUT_GATE_UP ? 1 : 0;
  p.out_mode = a.out_mode;
  p.out_f32 = static_cast<float*>(a.out_f32);
  const int32_t* offsets = a.offsets;
  const int32_t* pairs = a.pairs;
  const int32_t* active = a.active;
  const int32_t* n_active = a.n_active;
  void* out = a.out;
  p.x = static_cast<const __nv_bfloat16*>(x);
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
  p.nsteps = w->Kp / 128;
  // a 128-byte weight box per row and step: rows of at least 128 packed bytes
  if (w->Kp < 256) return set_error(MX_ERR_UNSUPPORTED, "MXFP4 experts need K > 128 (K = %d)", w->K);
  CUtensorMap wmap;
  const int KHp = w->Kp / 2;
  int rc = encode_tensor_map_2d(&wmap, w->bytes, CU_TENSOR_MAP_DATA_TYPE_UINT8, KHp,
                                static_cast<uint64_t>(w->E) * w->N, KHp, 128, 16, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != MX_OK) return rc;
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  static int smem_set[64];
  if (raise_smem_limit(reinterpret_cast<const void*>(moe_kernel), kMoeSmem, di, smem_set) != MX_OK)
    return MX_ERR_CUDA;
  cudaError_t e;
  const long long P = static_cast<long long>(T) * topk;
  const int zmax = static_cast<int>(P < w->E ? P : w->E);
  dim3 grid((w->N + kMoeRows - 1) / kMoeRows, zmax, 1);
  moe_kernel<<<grid, kMoeWarps * 32, kMoeSmem, stream>>>(wmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

}  // namespace mx
