// K-ROUTE (token -> expert grouping) and K-MOE (routed A16W4 expert GEMM).
//
// A16W4 product (a16w4 = vllm.models.minimax_m3.amd.specialized_decode.mono.a16w4,
// module text, dequant, step_mfma): every MXFP4 weight is its e2m1 value times
// the row's E8M0 block scale, multiplied by the bf16 token activations with f32
// accumulation.  On the 5th-generation tensor cores this is a block-scaled
// product of kind::mxf8f6f4 with an e2m1 A operand (the weight, its codes E8M0
// scale factors in tensor memory) and an e4m3 B operand: the bf16 activation
// enters as two MXFP8 pieces hi + lo (see act_pieces_kernel) whose products
// accumulate into the same f32 accumulator.  The MXFP8-activation variant (MXFP4 x MXFP8, the
// prefill form of the same layer) uses hi alone, which is exactly the per-token
// MXFP8 quantization of the activation.
//
// Routing is the plainest reading of "routed experts" (the pages show no
// router): pairs grouped by expert id, stable in (token, slot) order.

#include "mx_common.cuh"
#include "mx_internal.h"
#include "tc_common.cuh"

namespace mx {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

// Zero the bf16 rows [P, N] of the pairs in [p0, p1) whose id is not a valid
// expert: each warp finds the invalid ids among 32 pairs and writes each such
// row with all its lanes (16-byte stores when N % 8 == 0).  Called by every
// thread of the CTA.
MX_DEV void zero_invalid_rows(const int32_t* __restrict__ ids, int p0, int p1, int E,
                              __nv_bfloat16* __restrict__ out, int N) {
  const int lane = threadIdx.x & 31;
  for (int w0 = p0 + static_cast<int>(threadIdx.x & ~31u); w0 < p1; w0 += blockDim.x) {  // warp-uniform
    const int p = w0 + lane;
    const int e = p < p1 ? ids[p] : 0;
    unsigned m = __ballot_sync(0xffffffffu, p < p1 && (e < 0 || e >= E));
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      __nv_bfloat16* row = out + static_cast<long long>(w0 + src) * N;
      if ((N & 7) == 0) {
        uint4* r4 = reinterpret_cast<uint4*>(row);
        for (int n = lane; n < (N >> 3); n += 32) r4[n] = make_uint4(0u, 0u, 0u, 0u);
      } else {
        for (int n = lane; n < N; n += 32) row[n] = __float2bfloat16_rn(0.0f);
      }
    }
  }
}

// zero_out (optional): bf16 [P, zero_N] rows of the pairs whose id is not a
// valid expert are set to zero (they belong to no expert's list).  pass_off
// (optional): pass_off[e] = the number of passes of pw pairs the experts
// before e need, pass_off[E] the total.
__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ counts,
                 int32_t* __restrict__ offsets, int32_t* __restrict__ pairs,
                 int32_t* __restrict__ active, int32_t* __restrict__ n_active, int* dev_status,
                 __nv_bfloat16* __restrict__ zero_out, int zero_N, int32_t* __restrict__ pass_off, int pw) {
  extern __shared__ int rs[];
  pdl_launch_dependents();  // the next kernel may start its prologue; it waits for this grid
  int* cnt = rs;           // [E]
  int* base = rs + E;      // [E]
  int* wcnt = rs + 2 * E;  // [warps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = static_cast<int>(blockDim.x) >> 5;  // the launch sizes the CTA by the pairs
  const unsigned full = 0xffffffffu;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  int bad = 0;
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);  // integer counts: order-independent
    } else if (e != -1) {
      bad = 1;
    }
  }
  if (zero_out) zero_invalid_rows(ids, 0, P, E, zero_out, zero_N);
  bad = __syncthreads_or(bad);
  if (warp == 0) {  // exclusive scans of the counts (and passes), the ascending list of active experts
    int run = 0, arun = 0, prun = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? cnt[e] : 0;
      const int pc = pass_off && pw > 0 ? (c + pw - 1) / pw : 0;
      int incl = c, pincl = pc;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o);
        const int pv = __shfl_up_sync(full, pincl, o);
        if (lane >= o) {
          incl += v;
          pincl += pv;
        }
      }
      const unsigned am = __ballot_sync(full, c > 0);
      if (e < E) {
        counts[e] = c;
        offsets[e] = run + incl - c;
        base[e] = run + incl - c;
        if (pass_off) pass_off[e] = prun + pincl - pc;
        if (c > 0) active[arun + __popc(am & ((1u << lane) - 1u))] = e;
      }
      run += __shfl_sync(full, incl, 31);
      prun += __shfl_sync(full, pincl, 31);
      arun += __popc(am);
    }
    if (lane == 0) {
      offsets[E] = run;
      if (pass_off) pass_off[E] = prun;
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
      for (int w = 0; w < nwarps; ++w) s += wcnt[w * E + i];
      base[i] += s;
    }
    __syncthreads();
  }
}

// ---- the same routing for many pairs, on many CTAs (three launches): each
// CTA counts a chunk of kRouteChunk pairs, one CTA scans the per-chunk counts
// (giving each chunk its base in every expert's list), each CTA scatters its
// chunk stably.  The result is identical to route_kernel's.
constexpr int kRouteChunk = 1024;     // pairs a CTA of the many-CTA routing
constexpr int kRouteManyMin = 4096;   // pairs from which the many-CTA routing is used

__global__ void __launch_bounds__(kRouteThreads)
    route_count_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ ccount,
                       int* __restrict__ bad_flag, __nv_bfloat16* __restrict__ zero_out, int zero_N,
                       int32_t* __restrict__ inv) {
  extern __shared__ int rs[];  // cnt[E]
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += blockDim.x) rs[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kRouteChunk;
  const int p1 = p0 + kRouteChunk < P ? p0 + kRouteChunk : P;
  int bad = 0;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) {
      atomicAdd(&rs[e], 1);
    } else {
      if (e != -1) bad = 1;
      if (inv) inv[p] = -1;
    }
  }
  if (zero_out) zero_invalid_rows(ids, p0, p1, E, zero_out, zero_N);
  bad = __syncthreads_or(bad);
  if (bad && threadIdx.x == 0) atomicOr(bad_flag, 1);
  for (int e = threadIdx.x; e < E; e += blockDim.x) ccount[static_cast<long long>(blockIdx.x) * E + e] = rs[e];
}

// One CTA: per-expert totals, offsets, active list, pass offsets, status, and
// cbase[c][e] = offsets[e] + the pairs of expert e in chunks before c.
__global__ void __launch_bounds__(kRouteThreads)
    route_scan_kernel(const int32_t* __restrict__ ccount, int C, int E, int32_t* __restrict__ cbase,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                      int32_t* __restrict__ n_active, int* dev_status, const int* __restrict__ bad_flag,
                      int32_t* __restrict__ pass_off, int pw) {
  extern __shared__ int rs[];  // total[E]
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int t = 0;
    for (int c = 0; c < C; ++c) t += ccount[static_cast<long long>(c) * E + e];
    rs[e] = t;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned full = 0xffffffffu;
  if (warp == 0) {
    int run = 0, arun = 0, prun = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? rs[e] : 0;
      const int pc = pass_off && pw > 0 ? (c + pw - 1) / pw : 0;
      int incl = c, pincl = pc;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(full, incl, o);
        const int pv = __shfl_up_sync(full, pincl, o);
        if (lane >= o) {
          incl += v;
          pincl += pv;
        }
      }
      const unsigned am = __ballot_sync(full, c > 0);
      if (e < E) {
        counts[e] = c;
        offsets[e] = run + incl - c;
        if (pass_off) pass_off[e] = prun + pincl - pc;
        if (c > 0) active[arun + __popc(am & ((1u << lane) - 1u))] = e;
      }
      run += __shfl_sync(full, incl, 31);
      prun += __shfl_sync(full, pincl, 31);
      arun += __popc(am);
    }
    if (lane == 0) {
      offsets[E] = run;
      if (pass_off) pass_off[E] = prun;
      *n_active = arun;
      if (dev_status) *dev_status = *bad_flag ? MX_ERR_EXPERT_ID : MX_OK;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int b = offsets[e];
    for (int c = 0; c < C; ++c) {
      cbase[static_cast<long long>(c) * E + e] = b;
      b += ccount[static_cast<long long>(c) * E + e];
    }
  }
}

// Stable scatter of one chunk, blockDim pairs at a time (as in route_kernel).
__global__ void __launch_bounds__(kRouteThreads)
    route_scatter_kernel(const int32_t* __restrict__ ids, int P, int E, const int32_t* __restrict__ cbase,
                         int32_t* __restrict__ pairs, int32_t* __restrict__ inv) {
  extern __shared__ int rs[];
  int* base = rs;          // [E]
  int* wcnt = rs + E;      // [warps][E]
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned full = 0xffffffffu;
  for (int e = tid; e < E; e += blockDim.x) base[e] = cbase[static_cast<long long>(blockIdx.x) * E + e];
  __syncthreads();
  const int p0 = blockIdx.x * kRouteChunk;
  const int p1 = p0 + kRouteChunk < P ? p0 + kRouteChunk : P;
  for (int c0 = p0; c0 < p1; c0 += blockDim.x) {
    const int p = c0 + tid;
    const int e = p < p1 ? ids[p] : -1;
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
      if (inv) inv[p] = pos;
    }
    __syncthreads();
    for (int i = tid; i < E; i += blockDim.x) {
      int t = 0;
      for (int w = 0; w < kRouteWarps; ++w) t += wcnt[w * E + i];
      base[i] += t;
    }
    __syncthreads();
  }
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

// ---------------------------------------------------------------- activation pieces
//
// The routed pairs' activation rows, gathered in the expert-sorted pair order
// and cut into 32-wide MX blocks.  A16 (bf16 activations): each block is
// written as two MXFP8 pieces, hi = the per-token MXFP8 quantization of x and
// lo = the same quantization of the residual x - hi (exact in f32), so that
// hi + lo = x except where an element lies below the e4m3 normal range of its
// block's residual scale (|x - hi - lo| <= 2^-21.8 max|x| over the block).
// MXFP8 activations: hi only.  Row j of xh / xl is pair pairs[j]; its codes
// for K step s sit at cs[j][s][0..3] (hi) and cs[j][s][16..19] (lo): 16-byte
// rows of a tcgen05 scale-factor atom whose rows 0..15 scale the hi pieces of
// 16 pairs (B rows 0..15) and rows 16..31 their lo pieces (B rows 16..31).
__device__ __forceinline__ uint32_t mx_quant_f32x32(const float (&v)[32], uint4 (&out)[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
  const uint32_t code = mx_block_code(amax);
  const uint32_t ef = 254u - code;
  const float rescale = ef ? __uint_as_float(ef << 23) : __uint_as_float(0x00400000u);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = f32x2_to_e4m3x2(v[4 * i] * rescale, v[4 * i + 1] * rescale) |
           (f32x2_to_e4m3x2(v[4 * i + 2] * rescale, v[4 * i + 3] * rescale) << 16);
  out[0] = make_uint4(w[0], w[1], w[2], w[3]);
  out[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return code;
}

// One 32-value block of a bf16 activation row as MXFP8 pieces: the hi piece
// (qh, code ch) and, when lo, the residual x - hi quantized again (ql, cl).
// Blocks past K (valid = false): zero bytes and code 127.
MX_DEV void quant_pieces(const uint4 (&u)[4], bool valid, int lo, uint4 (&qh)[2], uint4 (&ql)[2], uint32_t& ch,
                         uint32_t& cl) {
  qh[0] = qh[1] = make_uint4(0u, 0u, 0u, 0u);
  ql[0] = ql[1] = qh[0];
  ch = 127u;
  cl = 127u;
  if (!valid) return;
  ch = mx_quant_bf16x32(u, qh);
  if (lo && ch != 255u) {
    const float scale = e8m0_to_f32(ch);
    const uint32_t hw[8] = {qh[0].x, qh[0].y, qh[0].z, qh[0].w, qh[1].x, qh[1].y, qh[1].z, qh[1].w};
    const uint32_t xw[16] = {u[0].x, u[0].y, u[0].z, u[0].w, u[1].x, u[1].y, u[1].z, u[1].w,
                             u[2].x, u[2].y, u[2].z, u[2].w, u[3].x, u[3].y, u[3].z, u[3].w};
    float r[32];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      // elements 2q, 2q + 1: bf16 -> f32 exactly, minus the dequantized hi piece
      const __half2 h = e4m3x2_to_f16x2(static_cast<uint16_t>(hw[q >> 1] >> (16 * (q & 1))));
      r[2 * q] = __uint_as_float(xw[q] << 16) - __low2float(h) * scale;
      r[2 * q + 1] = __uint_as_float(xw[q] & 0xffff0000u) - __high2float(h) * scale;
    }
    cl = mx_quant_f32x32(r, ql);
  }
}

// Rows past the routed pairs (slots with an invalid id are in no expert's
// list, so the list holds *n_pairs <= P entries) are left as they are: they
// only ever fill unused columns of a pass's last 32-row box.
// Wide passes (sfb != nullptr): instead of the 16-byte code rows, the codes
// go to the scale-factor atom of the row's pass: row r of pass c of expert e
// (r = its rank in the expert's list mod pw) is B row r (hi) and pw + r (lo),
// byte (m % 32) * 16 + (m / 32) * 4 + kb of atom [pass_off[e] + c][K step].
// The pieces of every (sorted position, block) (inv == nullptr: pairs [nv]
// lists the pair of each sorted position) or of every (activation row,
// block) (inv: the sorted position of each pair), split over the grid.
MX_DEV void act_pieces_body(const __nv_bfloat16* __restrict__ x, const int32_t* pairs, int nv, int P, int topk,
                            int x_per_pair, int K, int Kp, int lo, uint8_t* __restrict__ xh,
                            uint8_t* __restrict__ xl, uint8_t* __restrict__ cs, const int32_t* __restrict__ ids,
                            const int32_t* __restrict__ offsets, const int32_t* __restrict__ pass_off, int pw,
                            uint8_t* __restrict__ sfb, const int32_t* __restrict__ inv, int R) {
  const int KBp = Kp >> 5, KB = K >> 5, KT = Kp >> 7;
  // inv == nullptr: one thread a (sorted position, block), the position's
  // pair read from the list; else one thread a (activation row, block), the
  // row split once and written to every sorted position inv[] gives it
  const int fan = inv ? (x_per_pair ? 1 : topk) : 1;
  if (inv) nv = R;
  // 32-bit indices: the launcher checks P * Kp / 32 < 2^31
  const unsigned total = static_cast<unsigned>(inv ? R : (nv < P ? nv : P)) * static_cast<unsigned>(KBp);
  const int lane = threadIdx.x & 31;
  // warp-uniform loop (the code words below are gathered by shuffles): lanes
  // past the end take part but load and store nothing; total and the groups
  // of four lanes are multiples of 4, so a group is wholly in or out
  for (unsigned iw = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); iw < total; iw += gridDim.x * blockDim.x) {
    const unsigned i = iw + lane;
    const bool act = i < total;
    const unsigned ru = act ? i / static_cast<unsigned>(KBp) : 0u;
    const int b = act ? static_cast<int>(i - ru * static_cast<unsigned>(KBp)) : lane;
    long long src;
    if (inv) {
      src = ru;  // the activation row itself
    } else {
      const int pr = pairs[ru];
      src = x_per_pair ? pr : pr / topk;
    }
    uint4 u[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                  make_uint4(0u, 0u, 0u, 0u)};
    const bool valid = act && b < KB;  // padded K blocks: zero bytes, a finite code
    if (valid) {
      const uint4* sp = reinterpret_cast<const uint4*>(x + src * K + 32 * b);
#pragma unroll
      for (int q = 0; q < 4; ++q) u[q] = sp[q];
    }
    uint4 qh[2], ql[2];
    uint32_t ch, cl;
    quant_pieces(u, valid, lo, qh, ql, ch, cl);
    // the codes of blocks 4 g .. 4 g + 3 are 4 consecutive bytes of a scale
    // atom row (or of a code row): lane 4 g writes them as one word
    uint32_t wh = ch & 0xffu, wl = cl & 0xffu;
#pragma unroll
    for (int d = 1; d < 4; ++d) {
      wh |= (__shfl_down_sync(0xffffffffu, ch, d) & 0xffu) << (8 * d);
      wl |= (__shfl_down_sync(0xffffffffu, cl, d) & 0xffu) << (8 * d);
    }
    const bool leader = (b & 3) == 0;
    if (!act) continue;
    for (int f = 0; f < fan; ++f) {
      long long j;
      int pr;
      if (inv) {
        pr = static_cast<int>(ru) * fan + f;  // the pair
        j = inv[pr];
        if (j < 0) continue;                  // an invalid id: in no list
      } else {
        j = ru;
        pr = pairs[ru];
      }
      uint4* hp = reinterpret_cast<uint4*>(xh + j * Kp + 32 * b);
      hp[0] = qh[0];
      hp[1] = qh[1];
      if (lo) {
        uint4* lp = reinterpret_cast<uint4*>(xl + j * Kp + 32 * b);
        lp[0] = ql[0];
        lp[1] = ql[1];
      }
      if (sfb) {
        const int e = ids[pr];
        const int rank = static_cast<int>(j) - offsets[e];
        const int r = rank % pw;
        uint8_t* atom = sfb + (static_cast<long long>(pass_off[e] + rank / pw) * KT + (b >> 2)) * 512;
        if (leader) {
          *reinterpret_cast<uint32_t*>(atom + (r & 31) * 16 + (r >> 5) * 4) = wh;
          if (lo) *reinterpret_cast<uint32_t*>(atom + ((pw + r) & 31) * 16 + ((pw + r) >> 5) * 4) = wl;
        }
      } else if (leader) {
        uint8_t* cp = cs + (j * KT + (b >> 2)) * 32;
        *reinterpret_cast<uint32_t*>(cp) = wh;
        if (lo) *reinterpret_cast<uint32_t*>(cp + 16) = wl;
      }
    }
  }
}

__global__ void act_pieces_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pairs,
                                  const int32_t* __restrict__ n_pairs, int P, int topk, int x_per_pair, int K,
                                  int Kp, int lo, uint8_t* __restrict__ xh, uint8_t* __restrict__ xl,
                                  uint8_t* __restrict__ cs, const int32_t* __restrict__ ids,
                                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ pass_off, int pw,
                                  uint8_t* __restrict__ sfb, const int32_t* __restrict__ inv, int R) {
  pdl_launch_dependents();
  pdl_wait_prior_grid();  // the routing (and the activation, when a kernel wrote it) is complete
  act_pieces_body(x, pairs, inv ? R : *n_pairs, P, topk, x_per_pair, K, Kp, lo, xh, xl, cs, ids, offsets, pass_off,
                  pw, sfb, inv, R);
}

// Routing and activation pieces in one kernel for decode sizes (at most
// kRoutePairs pairs, narrow passes): every CTA sorts the ids in shared memory
// (the routing kernel's order: experts ascending, each expert's pairs in pair
// order), CTA 0 publishes the routing the expert GEMM and the finishing kernel
// read (offsets [E + 1], active, n_active, pairs, status) and zeroes the bf16
// rows [zero_N] of the pairs whose id is not an expert, and every CTA writes
// the pieces of its share of the sorted positions.  One launch less on the
// decode chain: on GB300 (E=256 N=4096 K=7168 top-8, T=1) the separate
// routing kernel kept the pieces waiting about 3.5 us.
constexpr int kRoutePairs = 64;
__global__ void __launch_bounds__(256) act_route_kernel(
    const int32_t* __restrict__ ids, int P, int E, int topk, const __nv_bfloat16* __restrict__ x, int x_per_pair,
    int K, int Kp, int lo, uint8_t* __restrict__ xh, uint8_t* __restrict__ xl, uint8_t* __restrict__ cs,
    int32_t* __restrict__ offsets, int32_t* __restrict__ pairs, int32_t* __restrict__ active,
    int32_t* __restrict__ n_active, int* dev_status, __nv_bfloat16* __restrict__ zero_out, int zero_N) {
  __shared__ int r_ids[kRoutePairs], r_pairs[kRoutePairs], r_act[kRoutePairs], r_off[kRoutePairs + 1];
  __shared__ unsigned r_bits[MX_MAX_EXPERTS / 32];
  __shared__ int r_na;
  // the ids and x are complete, and the previous call's kernels no longer read
  // the routing; only then may the expert GEMM start (it reads the ids and
  // the weights before its own dependency wait)
  pdl_wait_prior_grid();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < MX_MAX_EXPERTS / 32) r_bits[tid] = 0u;
  __syncthreads();
  bool valid = false, bad = false;
  if (tid < P) {
    const int e = ids[tid];
    valid = e >= 0 && e < E;
    bad = !valid && e != -1;
    r_ids[tid] = valid ? e : -1;
    if (valid) atomicOr(&r_bits[e >> 5], 1u << (e & 31));
  }
  const int n_valid = __syncthreads_count(valid);
  const int any_bad = __syncthreads_or(bad);
  if (warp == 0) {
    // the active experts in ascending order: lane l owns bit word l
    unsigned wb = lane < (E + 31) / 32 ? r_bits[lane] : 0u;
    const int c = __popc(wb);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int k = incl - c;
    while (wb) {
      r_act[k++] = lane * 32 + __ffs(wb) - 1;
      wb &= wb - 1;
    }
    const int na = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      r_na = na;
      r_off[na] = n_valid;
    }
  } else if (warp == 1 || warp == 2) {
    // sorted position of pair q: the valid pairs of smaller experts, then the
    // earlier pairs of its own
    const int q = tid - 32;
    if (q < P && r_ids[q] >= 0) {
      const int eq = r_ids[q];
      int below = 0, before = 0;
      for (int j = 0; j < P; ++j) {
        const int ej = r_ids[j];
        below += (ej >= 0 && ej < eq) ? 1 : 0;
        before += (j < q && ej == eq) ? 1 : 0;
      }
      r_pairs[below + before] = q;
      if (before == 0) {
        int a = __popc(r_bits[eq >> 5] & ((1u << (eq & 31)) - 1u));  // the expert's rank among the active
        for (int wd = 0; wd < (eq >> 5); ++wd) a += __popc(r_bits[wd]);
        r_off[a] = below;
      }
    }
  }
  __syncthreads();
  const int na = r_na;
  if (blockIdx.x == 0) {
    // offsets[e]: the valid pairs of the experts below e
    for (int e = tid; e <= E; e += blockDim.x) {
      int a = 0;
      for (int wd = 0; wd < (e >> 5); ++wd) a += __popc(r_bits[wd]);
      if ((e & 31) && (e >> 5) < MX_MAX_EXPERTS / 32) a += __popc(r_bits[e >> 5] & ((1u << (e & 31)) - 1u));
      offsets[e] = r_off[a];
    }
    for (int j = tid; j < n_valid; j += blockDim.x) pairs[j] = r_pairs[j];
    for (int a = tid; a < na; a += blockDim.x) active[a] = r_act[a];
    if (tid == 0) {
      *n_active = na;
      if (dev_status) *dev_status = any_bad ? MX_ERR_EXPERT_ID : MX_OK;
    }
    if (zero_out && warp == 7) {
      for (int w0 = 0; w0 < P; w0 += 32) {
        unsigned m = __ballot_sync(0xffffffffu, w0 + lane < P && r_ids[w0 + lane] < 0);
        while (m) {
          const int q = w0 + __ffs(m) - 1;
          m &= m - 1;
          for (int n = lane; n < zero_N; n += 32) zero_out[static_cast<long long>(q) * zero_N + n] = __float2bfloat16_rn(0.0f);
        }
      }
    }
  }
  act_pieces_body(x, r_pairs, n_valid, P, topk, x_per_pair, K, Kp, lo, xh, xl, cs, nullptr, nullptr, nullptr, 0,
                  nullptr, nullptr, 0);
}

// ---------------------------------------------------------------- expert GEMM
//
// Persistent CTAs walking (expert, 128-row tile) work items; 8 warps:
//   warp 0 (lane 0)  streams the weight tile, one K step (128 rows x 128 e2m1
//                    values, a contiguous 8 KB block) a stage: a TMA load with
//                    the 16U4_ALIGN16B data type writes it straight in the
//                    tensor core's e2m1 operand form (16 values = 8 packed
//                    bytes a 16-byte chunk, the other 8 bytes not written and
//                    not read, 128B swizzle), plus the step's 512-byte weight
//                    scale atom;
//   warp 2 (lane 0)  streams the B operand of the expert's next pass of
//                    pairs: their hi rows then (A16) their lo rows, 128 bytes
//                    of e4m3 a row for the K step (128B swizzle), and the scale
//                    atom of those rows;
//   warp 1 (lane 0)  allocates tensor memory and issues, per K step, the two
//                    scale copies and 4 block-scaled MMAs (kind::mxf8f6f4,
//                    scale_vec::1X, A e2m1, B e4m3, M = 128 weight rows,
//                    N = the B rows, K = 32): one f32 accumulator column a B
//                    row;
//   warps 4..7       read the accumulator (tcgen05.ld, one lane quarter each),
//                    add each pair's hi and lo columns and store bf16 /
//                    SiLU-and-mul / f32 per pair.
// Two pass widths.  Narrow (decode: a few pairs an expert): 32 B rows (16
// pairs with hi and lo, or 32 pairs hi only), the activation scale atom taken
// by TMA from the pairs' 16-byte code rows, two accumulators, three CTAs an
// SM.  Wide (prefill: hundreds of pairs an expert): 128 B rows (64 pairs with
// hi and lo, or 128 hi only), the scale atom of the pass laid out by the
// activation-pieces kernel and bulk-copied, one accumulator, two CTAs an SM.
constexpr uint32_t pow2_at_least(uint32_t v, uint32_t c = 32) { return c >= v ? c : pow2_at_least(v, 2 * c); }

// A third form for prefill when the weight has an even number of 128-row
// tiles (kMoePair): each work item is two adjacent row tiles multiplied by
// the same activation stage (8 MMAs a K step into two accumulators), so every
// activation byte brought from L2 feeds twice the tensor work.  Each tile's
// MMAs are issued by a thread of their own (warps 1 and 3): one thread issues
// a block-scaled MMA only about every 150 cycles (measured on GB300), about
// twice the tensor time of an M=128 N=128 K=32 MMA, so one issuer would leave
// the tensor core idle half the time.  One CTA an SM
// and 12 warps (8 epilogue warps, one a lane quarter of each accumulator); the
// epilogue copies its accumulator quarter to registers and releases it before
// the stores, so the next pass's MMAs overlap them.
//
// A fourth form for decode (kMoeNarrow16: at most kSplitMaxPairs pairs, or few
// pairs an expert): narrow
// passes of 16 B rows (8 pairs with hi and lo, or 16 hi only).  Its 2 KB
// activation stages leave room for four weight stages at three CTAs an SM
// instead of three (E=256 N=4096 K=7168 top-8 on GB300: the expert kernel
// alone 28.3 -> 26.9 us at T=1, calls 2-5 % faster at T=1..8).  Fewer,
// deeper CTAs do not help: two CTAs an SM with five or six weight stages ran
// 16-24 % slower, each CTA having one MMA issuer.
constexpr int kMoeNarrow = 0, kMoeWide = 1, kMoePair = 2, kMoeNarrow16 = 3;
constexpr int kEarlyPairs = 64;  // pairs the 16-row form can route itself (MoeParams::early)

template <int kMode>
struct MoeCfg {
  static constexpr bool kNarrow = kMode == kMoeNarrow || kMode == kMoeNarrow16;
  static constexpr bool kWide = !kNarrow;
  static constexpr int kATiles = kMode == kMoePair ? 2 : 1;    // 128-row weight tiles an item
  static constexpr int kBRows = kWide ? 128 : (kMode == kMoeNarrow16 ? 16 : 32);  // B rows a pass (MMA N)
  static constexpr int kWStages = kMode == kMoePair || kMode == kMoeNarrow16 ? 4 : 3;
  static constexpr int kXStages = kMode == kMoePair ? 4 : 3;  // the activation comes from L2
  // The weight ring's stage-empty barriers also free the activation stages:
  // activation stage g % X is free once the MMAs of step g - X completed,
  // which is phase (g - X) / W of weight barrier (g - X) % W (with X <= W it
  // cannot have run a phase further: that needs step g's activation).  So an
  // issuer makes one tcgen05.commit a K step instead of two.  Each tcgen05
  // instruction costs the single issuing thread issue time, and that time is
  // what bounds the prefill forms (measured on GB300, E=64 N=K=4096 T=4096
  // top-8: W4A8 572 -> 509 us, A16W4 1040 -> 905 us, the two-tile form going
  // from 5 activation stages to 4 for it; the 32-row narrow form from 5 to 3:
  // A16W4 T=64 101.6 -> 99.7 us).
  static_assert(kXStages <= kWStages, "activation stages are freed through the weight ring's barriers");
  static constexpr int kAccBufs = kWide ? 1 : 2;
  static constexpr int kCtasPerSm = kNarrow ? 3 : (kMode == kMoeWide ? 2 : 1);
  static constexpr int kThreads = kMode == kMoePair ? 384 : 256;
  static constexpr int kEpiWarps = 4 * kATiles;
  static constexpr int kWStage = kATiles * 128 * 128;         // e2m1 operand steps, 128B swizzle
  static constexpr int kXStage = kBRows * 128;                // B rows, 128B swizzle (1 KB aligned)
  static constexpr int kWOff = 0;
  static constexpr int kXOff = kWOff + kWStages * kWStage;
  static constexpr int kSfaOff = kXOff + kXStages * kXStage;  // kATiles weight scale atoms a weight stage
  static constexpr int kSfbOff = kSfaOff + kWStages * kATiles * 512;  // an activation scale atom a stage
  static constexpr int kBarOff = kSfbOff + kXStages * 512;
  static constexpr int kNumBars = 2 * kWStages + kXStages + 2 * kAccBufs;  // w full, w empty, x full, acc full, acc empty
  // tensor-memory slot, abort flag, the narrow passes' K ranges and items;
  // then (wide) the experts' pass offsets.  No static shared memory: it is
  // allocated in 1 KB units, and the four-stage decode form fits three CTAs an
  // SM only without it.
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kPoOff = kMiscOff + 16;
  // 16-row form routing itself (early): sorted pairs (u8), active experts
  // (u16), their first sorted positions and the valid count (u8)
  static constexpr int kEarlyOff = kPoOff + (kWide ? 4 * (MX_MAX_EXPERTS + 1) : 0);
  static constexpr int kEarlyBytes = kMode == kMoeNarrow16 ? kEarlyPairs + 2 * kEarlyPairs + kEarlyPairs + 2 : 0;
  static constexpr int kSmem = kEarlyOff + kEarlyBytes + 1024;  // + alignment slack
  static constexpr uint32_t kAccCols = kBRows;
  // tensor memory: the accumulator(s) | a (SFA 4 a tile, SFB 4 a tile) slot a
  // weight stage (each tile's issuer copies its own SFB)
  static constexpr uint32_t kSfSlot = kATiles == 2 ? 16 : 8;
  static constexpr uint32_t kTmemCols = pow2_at_least(kAccBufs * kATiles * kAccCols + kSfSlot * kWStages);
  static constexpr uint32_t kIdesc = mxf8_idesc_a(128, kBRows, kFmtE2M1);
};
constexpr int kWTx = 128 * 64;            // bytes the weight TMA writes a tile (the packed half of each chunk)
constexpr int kWidePairsA16 = 64, kWidePairsMx8 = 128;  // pairs a wide pass

struct MoeParams {
  const uint8_t* sfw;      // weight scale atoms [E, NT, KT, 512]
  const uint8_t* sfb;      // wide: activation scale atoms [passes, KT, 512]
  const int32_t* offsets;
  const int32_t* pairs;
  const int32_t* active;
  const int32_t* n_active;
  const int32_t* pass_off; // wide: first pass of each expert [E + 1]
  const int32_t* ids;      // early: the top-k ids [P]
  int early;               // 16-row form: route from ids before the grid-dependency wait (see moe_kernel)
  __nv_bfloat16* out;      // kMoeOutBf16: [T * topk, N]; kMoeOutSwiglu: [T * topk, N / 2]
  float* out_f32;          // kMoeOutF32: [T * topk, N]
  int N, KT, NT, E;
  int ksplit;              // narrow passes: at most this many K ranges an item (1: no split;
                           // the count itself is moe_split_for of the active experts)
  int P;                   // T * topk
  float* part;             // ksplit > 1: f32 partial sums [ranges, P, N]
  int32_t* split_out;      // ksplit > 1: CTA 0 writes the K ranges it chose here (for the finishing kernel)
  int lo;                  // 1: hi and lo activation pieces (A16), 0: hi only (MXFP8)
  int gate_up;             // weight rows interleaved gate / up in 8-row groups
  int out_mode;
};

// Packed row r of a gate / up interleaved weight -> its row in gate-then-up order.
MX_DEV int gate_up_row(int r, int N) {
  const int q = r >> 4, i = r & 15;
  return i < 8 ? 8 * q + i : (N >> 1) + 8 * q + i - 8;
}

MX_DEV float silu_f32(float v) { return v / (1.0f + expf(-v)); }

// Narrow passes: a work item is one K range of one group of `tiles` 128-row
// tiles of the a-th active expert, all its passes of pairs (items a-major,
// the K range fastest).  Wide passes
// (po = the experts' pass offsets): a work item is one pass of one tile group,
// items expert-major, then tile group, then pass, so the CTAs that read the
// same weight tiles for the passes of an expert run side by side and share
// them through L2.  Every role of a CTA walks the same items blockIdx.x,
// + gridDim.x, ...
struct Item {
  int e, o0, cnt, rt;
  int ch0, nch;  // the item's passes
  int npass;     // the passes of its expert
  int s0, s1;    // the item's K steps (narrow passes split K into ksplit ranges)
  int ks;        // ... the range's index
};

MX_DEV Item item_at(const MoeParams& p, int i, int tok, int tiles, const int* po, int S) {
  Item it;
  const int nti = p.NT / tiles;  // tile groups an expert (tiles = 2 needs NT even)
  if (po) {
    // the expert: the largest e with po[e] * nti <= i (po[E] * nti > i)
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (po[mid] * nti <= i) lo = mid; else hi = mid;
    }
    it.e = lo;
    it.npass = po[lo + 1] - po[lo];
    const int local = i - po[lo] * nti;
    const int g = local / it.npass;
    it.rt = g * tiles;
    it.ch0 = local - g * it.npass;
    it.nch = 1;
    it.o0 = p.offsets[it.e];
    it.cnt = p.offsets[it.e + 1] - it.o0;
    it.s0 = 0;
    it.s1 = p.KT;
    it.ks = 0;
    return it;
  }
  // narrow: items (active expert, tile group, K range), the K range fastest
  // (the ranges of a tile run side by side; numbered range-slowest instead, the
  // E=256 K=7168 top-8 decode calls ran 7-14 % slower on GB300)
  const int a = i / (nti * S);
  const int rem = i - a * nti * S;
  const int g = rem / S, ks = rem - g * S;
  it.s0 = ks * p.KT / S;
  it.s1 = (ks + 1) * p.KT / S;
  it.ks = ks;
  it.rt = g * tiles;  // the item's first 128-row tile
  it.e = p.active[a];
  it.o0 = p.offsets[it.e];
  it.cnt = p.offsets[it.e + 1] - it.o0;
  it.nch = (it.cnt + tok - 1) / tok;
  it.ch0 = 0;
  it.npass = it.nch;
  return it;
}

// 16-row form routing itself (early): item i as in item_at's narrow passes,
// the expert and its pairs from the CTA's shared-memory tables (eact: the
// active experts ascending; eoff: each one's first sorted position, then the
// valid count).
MX_DEV Item item_at_early(const MoeParams& p, int i, int tok, int S, const uint16_t* eact, const uint8_t* eoff) {
  Item it;
  const int nti = p.NT;
  const int a = i / (nti * S);
  const int rem = i - a * nti * S;
  const int g = rem / S, ks = rem - g * S;
  it.s0 = ks * p.KT / S;
  it.s1 = (ks + 1) * p.KT / S;
  it.ks = ks;
  it.rt = g;
  it.e = eact[a];
  it.o0 = eoff[a];
  it.cnt = eoff[a + 1] - it.o0;
  it.nch = (it.cnt + tok - 1) / tok;
  it.ch0 = 0;
  it.npass = it.nch;
  return it;
}

// One pair's output value y for weight row n (lane l of the warp holds row n).
MX_DEV void store_pair(const MoeParams& p, int pt, int n, int lane, float y) {
  if (p.out_mode == kMoeOutSwiglu) {
    // lane l (l % 16 < 8) holds gate row 8 (n / 16) + l % 16, lane l + 8 its up row
    const float u = __shfl_down_sync(0xffffffffu, y, 8);
    if ((lane & 15) < 8 && n < p.N)
      p.out[static_cast<long long>(pt) * (p.N >> 1) + (n >> 4) * 8 + (n & 15)] = __float2bfloat16_rn(silu_f32(y) * u);
  } else if (p.out_mode == kMoeOutF32) {
    if (n < p.N) p.out_f32[static_cast<long long>(pt) * p.N + n] = y;
  } else if (p.out_mode == kMoeOutBf16 && n < p.N) {
    const int nn = p.gate_up ? gate_up_row(n, p.N) : n;
    p.out[static_cast<long long>(pt) * p.N + nn] = __float2bfloat16_rn(y);
  }
}

// The K ranges an item of the narrow passes (1 .. kmax), from the number of
// (active expert, row tile) items and the CTAs that walk them (slots): the
// count that minimises the K steps of the busiest CTA, ceil(items S / slots)
// ranges of at most ceil(KT / S) steps each, plus 0.5 % of an item for each
// extra range (its accumulator switch, its partial sums and their final sum).
// Each range is charged at the longest one's length: CTA b takes items b,
// b + slots, ..., the K range fastest, so when slots is a multiple of S every
// CTA keeps one range index and the longer ranges of an uneven split land on
// the same CTAs.  Costs in 1/200 K steps; items * S and the rounds stay
// within 32 bits (items <= 512 experts x 2^16 row tiles), a cost within 38.
// The expert GEMM and the finishing kernel both evaluate it on the device from
// the routing's count of active experts, so the host never needs that count:
// one warp, lane S - 1 costing S, then a minimum over the lanes (ties to the
// smaller S), so no thread runs a chain of divisions.
MX_DEV int moe_split_for(unsigned items, unsigned slots, unsigned KT, int kmax, int lane) {
  const unsigned S = static_cast<unsigned>(lane) + 1u;
  unsigned long long key = ~0ull;
  if (S <= static_cast<unsigned>(kmax)) {
    const unsigned rounds = (items * S + slots - 1) / slots;
    const unsigned long long c =
        static_cast<unsigned long long>(rounds) * ((KT + S - 1) / S) * 200u + static_cast<unsigned long long>(KT) * (S - 1);
    key = (c << 5) | static_cast<unsigned>(lane);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
    key = other < key ? other : key;
  }
  return static_cast<int>(key & 31u) + 1;
}

// Split-K finish: each valid pair's output from the S f32 partial sums
// part [S, P, N] (S = moe_split_for of the active experts, read from where the
// GEMM wrote it),
// added in range order (deterministic), in the pass's output form.  Launched
// as a programmatic dependent of the expert GEMM; it does not release its own
// dependents early (measured on GB300: letting the next call's activation
// kernel launch at once was no faster, T=1 28.1 -> 28.4 us).  One thread 4
// consecutive output columns of a pair.  It sits on the decode call's critical
// path, so its dependent loads are few: the range count, the valid count and
// the pair's row in one round trip, then every range's partial sums at once.
constexpr int kFinishMaxSplit = 8;  // ranges the finishing kernel unrolls (>= kMaxKSplit)

__global__ void __launch_bounds__(256) moe_finish_kernel(const float* __restrict__ part,
                                                         const int32_t* __restrict__ split, int P, int N,
                                                         const int32_t* __restrict__ pairs,
                                                         const int32_t* __restrict__ n_valid, int out_mode,
                                                         int gate_up, __nv_bfloat16* __restrict__ out,
                                                         float* __restrict__ out_f32) {
  pdl_wait_prior_grid();
  const int cols = out_mode == kMoeOutSwiglu ? N / 2 : N;
  const int cols4 = (cols + 3) >> 2;
  const long long total = static_cast<long long>(P) * cols4;
  const long long PN = static_cast<long long>(P) * N;
  const bool vec = (N & 7) == 0;  // 16-byte partial rows, 8-byte bf16 / 16-byte f32 stores
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(idx / cols4), c = static_cast<int>(idx - static_cast<long long>(j) * cols4) * 4;
    // independent loads (pairs holds P entries; j < P)
    const int S = *split, nv = *n_valid, pt = pairs[j];
    if (S == 1) return;  // the GEMM did not split K and wrote the outputs itself
    if (j >= nv) continue;
    const float* src = part + static_cast<long long>(pt) * N;
    if (out_mode == kMoeOutSwiglu) {
      // packed rows 16 (c / 8) + c % 8 (gate) and 8 further on (up); 4
      // consecutive c stay inside one group of 8
      const int ng = (c >> 3) * 16 + (c & 7);
      float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec) {
        float4 pg[kFinishMaxSplit], pu[kFinishMaxSplit];
#pragma unroll
        for (int k = 0; k < kFinishMaxSplit; ++k)
          if (k < S) {
            pg[k] = *reinterpret_cast<const float4*>(src + k * PN + ng);
            pu[k] = *reinterpret_cast<const float4*>(src + k * PN + ng + 8);
          }
#pragma unroll
        for (int k = 0; k < kFinishMaxSplit; ++k)
          if (k < S) {
            g[0] += pg[k].x; g[1] += pg[k].y; g[2] += pg[k].z; g[3] += pg[k].w;
            u[0] += pu[k].x; u[1] += pu[k].y; u[2] += pu[k].z; u[3] += pu[k].w;
          }
        const __nv_bfloat162 a = __floats2bfloat162_rn(silu_f32(g[0]) * u[0], silu_f32(g[1]) * u[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(silu_f32(g[2]) * u[2], silu_f32(g[3]) * u[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&a);
        pk.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(out + static_cast<long long>(pt) * cols + c) = pk;
      } else {
        for (int e = 0; e < 4 && c + e < cols; ++e) {
          for (int k = 0; k < S; ++k) {
            g[e] += src[k * PN + ng + e];
            u[e] += src[k * PN + ng + e + 8];
          }
          out[static_cast<long long>(pt) * cols + c + e] = __float2bfloat16_rn(silu_f32(g[e]) * u[e]);
        }
      }
    } else {
      float y[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec) {
        float4 pv[kFinishMaxSplit];
#pragma unroll
        for (int k = 0; k < kFinishMaxSplit; ++k)
          if (k < S) pv[k] = *reinterpret_cast<const float4*>(src + k * PN + c);
#pragma unroll
        for (int k = 0; k < kFinishMaxSplit; ++k)
          if (k < S) {
            y[0] += pv[k].x; y[1] += pv[k].y; y[2] += pv[k].z; y[3] += pv[k].w;
          }
        if (out_mode == kMoeOutF32) {
          *reinterpret_cast<float4*>(out_f32 + static_cast<long long>(pt) * N + c) = make_float4(y[0], y[1], y[2], y[3]);
        } else {
          // a gate / up interleaved weight's rows c..c+3 stay consecutive in gate-then-up order
          const int oc = gate_up ? gate_up_row(c, N) : c;
          const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]), b = __floats2bfloat162_rn(y[2], y[3]);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&a);
          pk.y = *reinterpret_cast<const uint32_t*>(&b);
          *reinterpret_cast<uint2*>(out + static_cast<long long>(pt) * N + oc) = pk;
        }
      } else {
        for (int e = 0; e < 4 && c + e < cols; ++e) {
          for (int k = 0; k < S; ++k) y[e] += src[k * PN + c + e];
          if (out_mode == kMoeOutF32) out_f32[static_cast<long long>(pt) * N + c + e] = y[e];
          else out[static_cast<long long>(pt) * N + (gate_up ? gate_up_row(c + e, N) : c + e)] = __float2bfloat16_rn(y[e]);
        }
      }
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(MoeCfg<kMode>::kThreads, MoeCfg<kMode>::kCtasPerSm)
    moe_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xhmap,
               const __grid_constant__ CUtensorMap xlmap, const __grid_constant__ CUtensorMap csmap,
               const MoeParams p) {
  using C = MoeCfg<kMode>;
  constexpr bool kWide = C::kWide;
  constexpr int kT = C::kATiles;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok = C::kBRows >> p.lo;  // pairs a pass

  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* wempty = wfull + C::kWStages;
  uint64_t* xfull = wempty + C::kWStages;
  uint64_t* accfull = xfull + C::kXStages;       // [kAccBufs]
  uint64_t* accempty = accfull + C::kAccBufs;    // [kAccBufs]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  int* s_items = reinterpret_cast<int*>(tmem_slot + 2);  // narrow: [K ranges an item, items]

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kWStages; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], kT);    // tcgen05.commit of each tile's issuer
    }
    for (int i = 0; i < C::kXStages; ++i) mbar_init(&xfull[i], 1);
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&accfull[i], kT);   // tcgen05.commit of each tile's issuer
      mbar_init(&accempty[i], C::kEpiWarps);  // one arrival an epilogue warp
    }
    *abort_flag = 0u;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next kernel may start its prologue once every CTA holds its tensor
  // memory (a dependent grid then never takes columns this grid waits for)
  pdl_launch_dependents();
  // 16-row form, early: this grid starts only once the activation kernel
  // before it has passed its own dependency wait, so the ids and the weights
  // are complete; the routing is made here from the ids and the weights
  // stream at once, and only the activation producer waits for the pieces
  // (measured on GB300, E=256 N=4096 K=7168 top-8 T=1: the first weight stage
  // had landed ~4 us after the wait, behind the routing's reads)
  uint8_t* epairs = smem + C::kEarlyOff;                                        // [64]
  uint16_t* eact = reinterpret_cast<uint16_t*>(smem + C::kEarlyOff + kEarlyPairs);  // [64]
  uint8_t* eoff = smem + C::kEarlyOff + 3 * kEarlyPairs;                        // [65]
  const bool early = kMode == kMoeNarrow16 && p.early;
  int na_early = 0;
  if (early) {
    // the routing kernel's order, built in weight stage 0 (no TMA has written
    // it yet): ids (-1: invalid) and the used experts' bit set, then the tables
    int16_t* eids = reinterpret_cast<int16_t*>(smem + C::kWOff);
    unsigned* ebits = reinterpret_cast<unsigned*>(smem + C::kWOff + 2 * kEarlyPairs);
    if (threadIdx.x < MX_MAX_EXPERTS / 32) ebits[threadIdx.x] = 0u;
    __syncthreads();
    bool valid = false;
    if (threadIdx.x < kEarlyPairs) {
      const int e = threadIdx.x < p.P ? p.ids[threadIdx.x] : -1;
      valid = e >= 0 && e < p.E;
      eids[threadIdx.x] = static_cast<int16_t>(valid ? e : -1);
      if (valid) atomicOr(&ebits[e >> 5], 1u << (e & 31));
    }
    const int n_valid = __syncthreads_count(valid);
    if (warp == 0) {
      // the active experts ascending: lane l owns bit word l
      unsigned wb = lane < MX_MAX_EXPERTS / 32 ? ebits[lane] : 0u;
      const int c = __popc(wb);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int k = incl - c;
      while (wb) {
        eact[k++] = static_cast<uint16_t>(lane * 32 + __ffs(wb) - 1);
        wb &= wb - 1u;
      }
      if (lane == 31) eoff[incl] = static_cast<uint8_t>(n_valid);
    } else if (warp == 1 || warp == 2) {
      // pair q's sorted position: the valid pairs of smaller experts, then its
      // expert's earlier pairs
      const int q = threadIdx.x - 32;
      const int eq = eids[q];
      if (eq >= 0) {
        int below = 0, before = 0;
        for (int j = 0; j < p.P; ++j) {
          const int ej = eids[j];
          below += (ej >= 0 && ej < eq) ? 1 : 0;
          before += (j < q && ej == eq) ? 1 : 0;
        }
        epairs[below + before] = static_cast<uint8_t>(q);
        if (before == 0) {
          int a = __popc(ebits[eq >> 5] & ((1u << (eq & 31)) - 1u));  // the expert's rank among the active
          for (int wd = 0; wd < (eq >> 5); ++wd) a += __popc(ebits[wd]);
          eoff[a] = static_cast<uint8_t>(below);
        }
      }
    }
    fence_proxy_async_smem();  // stage 0's temporaries before the weight TMA overwrites them
    __syncthreads();
    if (warp == 0) {
      int na = lane < MX_MAX_EXPERTS / 32 ? __popc(ebits[lane]) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) na += __shfl_xor_sync(0xffffffffu, na, o);
      na_early = na;
    }
  } else {
    pdl_wait_prior_grid();  // the routing and the activation pieces are complete
  }
  // wide passes: the experts' pass offsets in shared memory (items are found by
  // a binary search over them)
  int* po_s = reinterpret_cast<int*>(smem + C::kPoOff);
  const int* po = nullptr;
  if (kWide) {
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) po_s[e] = p.pass_off[e];
    po = po_s;
  }
  // narrow passes: the K ranges an item, and the items (CTAs past the last
  // item go straight to the exit)
  if (!kWide && warp == 0) {
    const int na = early ? na_early : *p.n_active;
    const int split = p.ksplit == 1 ? 1 : moe_split_for(na * (p.NT / kT), gridDim.x, p.KT, p.ksplit, lane);
    if (lane == 0) {
      if (p.ksplit > 1 && blockIdx.x == 0) *p.split_out = split;
      s_items[0] = split;
      s_items[1] = na * (p.NT / kT) * split;
    }
  }
  __syncthreads();
  const int S = kWide ? 1 : s_items[0];
  const int n_items = kWide ? po_s[p.E] * (p.NT / kT) : s_items[1];
  auto get_item = [&](int i) -> Item {
    return early ? item_at_early(p, i, tok, S, eact, eoff) : item_at(p, i, tok, kT, po, S);
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ weight producer
    tma_prefetch_desc(&wmap);
    int g = 0;
    for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x) {
      const Item it = get_item(i);
      // a weight tile read once streams past L2; read again (more than one
      // pass of pairs) it is kept
      const uint64_t pol = it.npass > 1 ? policy_evict_last() : policy_evict_first();
      const long long tile = static_cast<long long>(it.e) * p.NT + it.rt;  // the item's first tile
      for (int ch = it.ch0; ch < it.ch0 + it.nch && !*abort_flag; ++ch) {
        for (int s = it.s0; s < it.s1; ++s, ++g) {
          const int st = g % C::kWStages;
          if (!mbar_wait(&wempty[st], ((g / C::kWStages) & 1u) ^ 1u)) { *abort_flag = 1u; break; }
          mbar_arrive_expect_tx(&wfull[st], kT * (kWTx + 512));
#pragma unroll
          for (int t = 0; t < kT; ++t) {
            // tile (tile + t): its K step s is 128-value row (tile + t) * KT * 128 + 128 s
            const int row0 = static_cast<int>((tile + t) * p.KT * 128);
            tma_load_2d(smem + C::kWOff + st * C::kWStage + t * 16384, &wmap, &wfull[st], 0, row0 + s * 128, pol);
            bulk_load(smem + C::kSfaOff + (st * kT + t) * 512, p.sfw + ((tile + t) * p.KT + s) * 512, 512,
                      &wfull[st]);
          }
        }
      }
    }
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------------------ activation producer
    if (early) pdl_wait_prior_grid();  // the activation pieces are complete
    tma_prefetch_desc(&xhmap);
    if (!kWide) tma_prefetch_desc(&csmap);
    if (p.lo) tma_prefetch_desc(&xlmap);
    const uint64_t pol = policy_evict_last();  // every row tile of the expert reads them
    const uint32_t tx = kWide ? C::kBRows * 128 + 512 : C::kBRows * (128 + 16);
    int g = 0;
    for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x) {
      const Item it = get_item(i);
      for (int ch = it.ch0; ch < it.ch0 + it.nch && !*abort_flag; ++ch) {
        const int row0 = it.o0 + ch * tok;
        for (int s = it.s0; s < it.s1; ++s, ++g) {
          const int st = g % C::kXStages;
          // the MMAs of step g - X have completed (weight ring barrier of that step)
          if (g >= C::kXStages &&
              !mbar_wait(&wempty[(g - C::kXStages) % C::kWStages], ((g - C::kXStages) / C::kWStages) & 1u)) {
            *abort_flag = 1u;
            break;
          }
          uint8_t* dst = smem + C::kXOff + st * C::kXStage;
          uint8_t* atom = smem + C::kSfbOff + st * 512;
          mbar_arrive_expect_tx(&xfull[st], tx);
          // hi rows of the pass's pairs, then (A16) their lo rows
          tma_load_2d(dst, &xhmap, &xfull[st], s * 128, row0, pol);
          if (p.lo) tma_load_2d(dst + tok * 128, &xlmap, &xfull[st], s * 128, row0, pol);
          if (kWide) {
            bulk_load(atom, p.sfb + (static_cast<long long>(p.pass_off[it.e] + ch) * p.KT + s) * 512, 512,
                      &xfull[st]);
          } else {
            tma_load_2d(atom, &csmap, &xfull[st], s * 32, row0, pol);
            if (p.lo) tma_load_2d(atom + tok * 16, &csmap, &xfull[st], s * 32 + 16, row0, pol);
          }
        }
      }
    }
  } else if ((warp == 1 || (kT == 2 && warp == 3)) && lane == 0) {
    // ------------------------------------------------------------ MMA issuers
    // warp 1 issues tile 0's MMAs, warp 3 (two-tile items) tile 1's, each into
    // its own accumulator with its own scale copies
    const int t = warp == 1 ? 0 : 1;
    int gw = 0, gx = 0, gp = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      const Item it = get_item(i);
      for (int ch = it.ch0; ch < it.ch0 + it.nch && ok; ++ch, ++gp) {
        const int buf = gp % C::kAccBufs;  // the epilogue drains the other accumulator (narrow)
        if (!mbar_wait(&accempty[buf], ((gp / C::kAccBufs) & 1u) ^ 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(buf * kT) * C::kAccCols;
        for (int s = it.s0; s < it.s1; ++s, ++gw, ++gx) {
          const int ws = gw % C::kWStages, xs = gx % C::kXStages;
          if (!mbar_wait(&wfull[ws], (gw / C::kWStages) & 1u) ||
              !mbar_wait(&xfull[xs], (gx / C::kXStages) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // scale slot: SFA of each tile (4 columns each), then SFB once a tile
          const uint32_t sfc = tmem + C::kAccBufs * kT * C::kAccCols + static_cast<uint32_t>(ws) * C::kSfSlot;
          const uint32_t sfb = sfc + 4 * kT + 4 * t;
          tc_cp_sf(sfc + 4 * t, sf_desc(smem_u32(smem + C::kSfaOff + (ws * kT + t) * 512)));
          tc_cp_sf(sfb, sf_desc(smem_u32(smem + C::kSfbOff + xs * 512)));
          const uint64_t bdesc = sw128_desc(smem_u32(smem + C::kXOff + xs * C::kXStage));
          const uint64_t adesc = sw128_desc(smem_u32(smem + C::kWOff + ws * C::kWStage + t * 16384));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t id = C::kIdesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
            tc_mma_mxf8(acc + t * C::kAccCols, adesc + 2 * k, bdesc + 2 * k, id, sfc + 4 * t, sfb,
                        (s != it.s0 || k != 0) ? 1u : 0u);
          }
          tc_commit(&wempty[ws]);  // frees this step's weight stage and (X steps on) its activation stage
        }
        if (ok) tc_commit(&accfull[buf]);
      }
    }
    if (!ok) *abort_flag = 1u;
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // tensor-memory lane quarter: rows 32 q .. 32 q + 31
    const int et = (warp - 4) >> 2;    // the item's tile this warp drains
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(et) * C::kAccCols;
    int gp = 0;
    for (int i = blockIdx.x; i < n_items && !*abort_flag; i += gridDim.x) {
      const Item it = get_item(i);
      const int n = (it.rt + et) * 128 + q * 32 + lane;
      for (int ch = it.ch0; ch < it.ch0 + it.nch; ++ch, ++gp) {
        const int buf = gp % C::kAccBufs;
        const int ntok = it.cnt - ch * tok < tok ? it.cnt - ch * tok : tok;
        const int* prow = p.pairs + it.o0 + ch * tok;  // this pass's pairs
        if (!mbar_wait(&accfull[buf], (gp / C::kAccBufs) & 1u)) { *abort_flag = 1u; break; }
        tc_fence_after();
        const uint32_t acc = lane_base + static_cast<uint32_t>(buf * kT) * C::kAccCols;
        if (!kWide) {
          // A16: columns 0 .. kB/2 - 1 hi pieces, then their lo pieces; MXFP8: kB pairs
          constexpr int kB = C::kBRows;
          uint32_t v[kB];
          if constexpr (kB == 32) {
            tmem_ld32(acc, v);
          } else {
            tmem_ld16_async(acc, v);
            tmem_wait_ld();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[buf]);  // a later pass may overwrite it
          const int pr = lane >= ntok ? -1 : (early ? epairs[it.o0 + ch * tok + lane] : prow[lane]);
          if (p.lo) {
#pragma unroll
            for (int t = 0; t < kB / 2; ++t)
              v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(v[kB / 2 + t]));
          }
          if (S > 1) {
            // split K: this K range's f32 sums; the finishing kernel adds the ranges
            float* part = p.part + static_cast<long long>(it.ks) * p.P * p.N + n;
#pragma unroll
            for (int t = 0; t < kB; ++t) {
              if (t >= ntok) break;  // warp-uniform
              const int pt = __shfl_sync(0xffffffffu, pr, t);
              if (n < p.N) part[static_cast<long long>(pt) * p.N] = __uint_as_float(v[t]);
            }
          } else {
#pragma unroll
            for (int t = 0; t < kB; ++t) {
              if (t >= ntok) break;  // warp-uniform
              store_pair(p, __shfl_sync(0xffffffffu, pr, t), n, lane, __uint_as_float(v[t]));
            }
          }
        } else if (kMode == kMoePair) {
          // the whole quarter (128 columns: 128 pairs, or 64 hi | 64 lo) to
          // registers, release the accumulator, then the stores
          uint32_t v[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_async(acc + static_cast<uint32_t>(c * 32), v + 32 * c);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[buf]);  // the next pass may overwrite it
          if (p.lo) {
#pragma unroll
            for (int t = 0; t < 64; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(v[64 + t]));
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c * 32 >= ntok) break;  // warp-uniform
            const int pr = c * 32 + lane < ntok ? prow[c * 32 + lane] : -1;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              if (c * 32 + t >= ntok) break;  // warp-uniform
              store_pair(p, __shfl_sync(0xffffffffu, pr, t), n, lane, __uint_as_float(v[c * 32 + t]));
            }
          }
        } else {
          // 32 pairs at a time: hi columns 32 c.., (A16) lo columns tok + 32 c..
          for (int c = 0; c * 32 < ntok; ++c) {
            uint32_t v[32];
            tmem_ld32(acc + static_cast<uint32_t>(c * 32), v);
            if (p.lo) {
              uint32_t vl[32];
              tmem_ld32(acc + static_cast<uint32_t>(tok + c * 32), vl);
#pragma unroll
              for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(vl[t]));
            }
            const int pr = c * 32 + lane < ntok ? prow[c * 32 + lane] : -1;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              if (c * 32 + t >= ntok) break;  // warp-uniform
              store_pair(p, __shfl_sync(0xffffffffu, pr, t), n, lane, __uint_as_float(v[t]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&accempty[buf]);  // the next pass may overwrite it
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

unsigned int take_error_flags_moe() { return take_tu_error_flags(); }

cudaError_t launch_route(const int32_t* ids, int T, int topk, int E, int32_t* counts,
                         int32_t* offsets, int32_t* pairs, int32_t* active, int32_t* n_active,
                         int* dev_status, cudaStream_t stream, void* zero_out, int zero_N, int32_t* pass_off,
                         int pw) {
  // one CTA, as many warps as a pass of pairs needs (a warp's count row of E
  // entries is zeroed and summed every pass: few pairs, few warps)
  const int P = T * topk;
  const int threads = P <= 128 ? 128 : (P <= 256 ? 256 : (P <= 512 ? 512 : kRouteThreads));
  const int smem = (2 * E + (threads / 32) * E) * static_cast<int>(sizeof(int));
  cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (2 * E + kRouteWarps * E) * static_cast<int>(sizeof(int)));
  if (e != cudaSuccess) return e;
  route_kernel<<<1, threads, smem, stream>>>(ids, T * topk, E, counts, offsets, pairs, active,
                                                   n_active, dev_status,
                                                   static_cast<__nv_bfloat16*>(zero_out), zero_N, pass_off, pw);
  return cudaGetLastError();
}

int route_many_writes_inv(long long P) { return P > kRouteManyMin ? 1 : 0; }

size_t route_scratch_bytes(long long P, int E) {
  const long long C = (P + kRouteChunk - 1) / kRouteChunk;
  return static_cast<size_t>(2 * C * E + 4) * sizeof(int32_t);
}

cudaError_t launch_route_many(const int32_t* ids, int T, int topk, int E, int32_t* counts, int32_t* offsets,
                              int32_t* pairs, int32_t* active, int32_t* n_active, int* dev_status,
                              cudaStream_t stream, void* zero_out, int zero_N, int32_t* pass_off, int pw,
                              void* scratch, int32_t* inv) {
  const int P = T * topk;
  if (P <= kRouteManyMin)
    return launch_route(ids, T, topk, E, counts, offsets, pairs, active, n_active, dev_status, stream, zero_out,
                        zero_N, pass_off, pw);
  const int C = (P + kRouteChunk - 1) / kRouteChunk;
  int32_t* ccount = static_cast<int32_t*>(scratch);
  int32_t* cbase = ccount + static_cast<long long>(C) * E;
  int* bad = reinterpret_cast<int*>(cbase + static_cast<long long>(C) * E);
  cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int smem1 = E * static_cast<int>(sizeof(int));
  const int smem3 = (E + kRouteWarps * E) * static_cast<int>(sizeof(int));
  if ((e = cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem3)) !=
      cudaSuccess)
    return e;
  route_count_kernel<<<C, kRouteThreads, smem1, stream>>>(ids, P, E, ccount, bad,
                                                          static_cast<__nv_bfloat16*>(zero_out), zero_N, inv);
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kRouteThreads, 1, 1);
  cfg.dynamicSmemBytes = smem1;
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, route_scan_kernel, static_cast<const int32_t*>(ccount), C, E, cbase, counts,
                              offsets, active, n_active, dev_status, static_cast<const int*>(bad), pass_off, pw)) !=
      cudaSuccess)
    return e;
  cfg.gridDim = dim3(C, 1, 1);
  cfg.dynamicSmemBytes = smem3;
  return cudaLaunchKernelEx(&cfg, route_scatter_kernel, ids, P, E, static_cast<const int32_t*>(cbase), pairs, inv);
}

cudaError_t launch_combine(const float* y2, const int32_t* ids, const float* wts, int T, int topk, int E, int H,
                           void* out, cudaStream_t stream) {
  const long long total = static_cast<long long>(T) * (H / 4);
  combine_kernel<<<blocks_for(total, 256), 256, 0, stream>>>(y2, ids, wts, T, topk, E, H,
                                                             static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

// Activation pieces of P pairs: xh [P + 128, Kp] | xl [P + 128, Kp] | codes
// [P + 128, Kp/128, 32] (narrow passes) | wide-pass scale atoms [P/64 + E + 1,
// Kp/128, 512]; each region 256-byte aligned (spare rows: the last pass of
// pairs loads a full box).
constexpr int kSpareRows = 128;
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
static size_t act_region(long long P, int Kp) { return align256(static_cast<size_t>(P + kSpareRows) * Kp); }
static size_t act_codes(long long P, int Kp) {
  return align256(static_cast<size_t>(P + kSpareRows) * (Kp / 128) * 32);
}
static size_t act_atoms(long long P, int Kp, int E) {
  return align256(static_cast<size_t>(P / kWidePairsA16 + E + 1) * (Kp / 128) * 512);
}
size_t moe_act_bytes(long long P, int Kp, int E) { return 2 * act_region(P, Kp) + act_codes(P, Kp) + act_atoms(P, Kp, E); }

// Split K of the narrow passes: at most kMaxKSplit ranges, for at most
// kSplitMaxPairs pairs (the decode sizes whose few experts leave SM slots idle).
constexpr int kMaxKSplit = 8, kSplitMaxPairs = 64;
static_assert(kMaxKSplit <= 32, "the split choice costs one count a lane");
static_assert(kMaxKSplit <= kFinishMaxSplit, "the finishing kernel unrolls every range");
static_assert(kEarlyPairs >= kSplitMaxPairs && kEarlyPairs == 64, "the 16-row form routes its pairs with two ballots");
size_t moe_part_bytes(long long P, int N) {
  return P <= kSplitMaxPairs ? static_cast<size_t>(kMaxKSplit) * P * N * sizeof(float) : 0;
}

int moe_route_in_act(long long P, int E, int lo) { return P >= 1 && P <= kRoutePairs && moe_wide_pass(P, E, lo) == 0; }

// Pairs a wide pass, or 0 for narrow passes: wide once the experts average at
// least half a wide pass of pairs.
int moe_wide_pass(long long P, int E, int lo) {
  const int pw = lo ? kWidePairsA16 : kWidePairsMx8;
  const long long experts = P < E ? P : E;
  return experts > 0 && P >= experts * (pw / 2) ? pw : 0;
}

// Persistent grid of the expert GEMM: kCtasPerSm CTAs an SM (what shared and
// tensor memory allow), never more than the largest possible number of work
// items (narrow: every one of the at most min(P, E) experts split into kmax
// ranges; wide: one pass an item, the passes numbering at most P / pw + min(P, E)).
template <int kMode>
static int moe_grid(long long P, int E, int kmax, int NT, int pw, const DeviceInfo& di) {
  using C = MoeCfg<kMode>;
  const long long zmax = P < E ? P : E;
  const long long items = (C::kWide ? P / pw + zmax : zmax * kmax) * (NT / C::kATiles);
  const long long slots = static_cast<long long>(C::kCtasPerSm) * di.sm_count;
  return static_cast<int>(items < slots ? items : slots);
}

template <int kMode>
static int launch_moe_gemm(const MoeLaunch& a, const MoeParams& p, uint8_t* xh, uint8_t* xl, uint8_t* cs,
                           cudaLaunchConfig_t cfg) {
  using C = MoeCfg<kMode>;
  constexpr bool kWide = C::kWide;
  static_assert(C::kSmem <= 227 * 1024 && C::kTmemCols <= 512 && C::kXStage % 1024 == 0, "expert kernel budget");
  static_assert(C::kAccBufs * C::kATiles * C::kAccCols + C::kSfSlot * C::kWStages <= C::kTmemCols, "tmem");
  const mx_packed_weight* w = a.w;
  const long long P = static_cast<long long>(a.T) * a.topk;
  const int Kp = w->Kp, KT = Kp / 128;
  const uint64_t rows = static_cast<uint64_t>(P + kSpareRows);
  const uint32_t tok = static_cast<uint32_t>(C::kBRows >> a.lo);  // rows a box
  CUtensorMap wmap, xhmap, xlmap, csmap;
  // the packed tiles as rows of 128 e2m1 values (64 bytes), unpacked by the TMA
  const uint64_t wrows = static_cast<uint64_t>(w->E) * p.NT * KT * 128;
  int rc = encode_tensor_map_2d(&wmap, w->bytes, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 128, wrows, 64, 128, 128,
                                CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == MX_OK)
    rc = encode_tensor_map_2d(&xhmap, xh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Kp, rows, Kp, 128, tok,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == MX_OK)
    rc = encode_tensor_map_2d(&xlmap, xl, CU_TENSOR_MAP_DATA_TYPE_UINT8, Kp, rows, Kp, 128, tok,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == MX_OK)
    rc = encode_tensor_map_2d(&csmap, cs, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(KT) * 32, rows,
                              static_cast<uint64_t>(KT) * 32, 16, kWide ? 16 : tok, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != MX_OK) return rc;
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  static int smem_set[64];
  if (raise_smem_limit(reinterpret_cast<const void*>(moe_kernel<kMode>), C::kSmem, di, smem_set) != MX_OK)
    return MX_ERR_CUDA;
  const int grid = moe_grid<kMode>(P, w->E, p.ksplit, p.NT, a.wide_pass, di);
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_kernel<kMode>, wmap, xhmap, xlmap, csmap, p);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

int launch_moe(const MoeLaunch& a, cudaStream_t stream) {
  const mx_packed_weight* w = a.w;
  const long long P = static_cast<long long>(a.T) * a.topk;
  const int Kp = w->Kp, KT = Kp / 128;
  if (!w->sf) return set_error(MX_ERR_ARG, "the E2M1 weight has no scale atoms (pack it with mx_pack_weights)");
  if (!a.act || a.act_bytes < moe_act_bytes(P, Kp, w->E))
    return set_error(MX_ERR_WORKSPACE, "expert activation workspace of %zu bytes, needs %zu", a.act_bytes,
                     moe_act_bytes(P, Kp, w->E));
  const bool wide = a.wide_pass > 0;
  const int NT = (w->N + 127) / 128;
  if (wide && (!a.pass_off || !a.ids || a.wide_pass != moe_wide_pass(P, w->E, a.lo)))
    return set_error(MX_ERR_ARG, "wide expert passes need the routing's pass offsets");
  uint8_t* xh = static_cast<uint8_t*>(a.act);
  uint8_t* xl = xh + act_region(P, Kp);
  uint8_t* cs = xl + act_region(P, Kp);
  uint8_t* sfb = cs + act_codes(P, Kp);
  if (P * (Kp / 32) >= (1LL << 31))
    return set_error(MX_ERR_UNSUPPORTED, "T * topk * K / 32 = %lld exceeds 2^31", P * (Kp / 32));
  // with the inverse map, one thread a block of each activation row (tokens,
  // or pairs for a down projection); else one a block of each sorted pair
  const long long R = a.inv ? (a.x_per_pair ? P : a.T) : P;
  const long long nblk = R * (Kp / 32);
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks_for(nblk, 256)), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = &pdl;
  cfg.numAttrs = a.no_pdl ? 0 : 1;
  cudaError_t e;
  if (a.route_in_act) {
    // decode sizes: the routing made by the pieces kernel itself
    if (!moe_route_in_act(P, w->E, a.lo) || !a.ids || !a.route.offsets || !a.route.pairs || !a.route.active ||
        !a.route.n_active)
      return set_error(MX_ERR_ARG, "routing in the activation kernel needs <= %d pairs and its outputs", kRoutePairs);
    e = cudaLaunchKernelEx(&cfg, act_route_kernel, static_cast<const int32_t*>(a.ids), static_cast<int>(P), w->E,
                           a.topk, static_cast<const __nv_bfloat16*>(a.x), a.x_per_pair, w->K, Kp, a.lo, xh, xl, cs,
                           a.route.offsets, a.route.pairs, a.route.active, a.route.n_active, a.route.dev_status,
                           static_cast<__nv_bfloat16*>(a.route.zero_out), a.route.zero_N);
  } else {
    e = cudaLaunchKernelEx(&cfg, act_pieces_kernel, static_cast<const __nv_bfloat16*>(a.x),
                           static_cast<const int32_t*>(a.pairs), static_cast<const int32_t*>(a.offsets + w->E),
                           static_cast<int>(P), a.topk, a.x_per_pair, w->K, Kp, a.lo, xh, xl, cs,
                           static_cast<const int32_t*>(a.ids), static_cast<const int32_t*>(a.offsets),
                           static_cast<const int32_t*>(a.pass_off), a.wide_pass, wide ? sfb : nullptr,
                           static_cast<const int32_t*>(a.inv), static_cast<int>(R));
  }
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "activation pieces launch: %s", cudaGetErrorString(e));

  MoeParams p = {};
  p.sfw = w->sf;
  p.sfb = sfb;
  p.offsets = a.offsets;
  p.pairs = a.pairs;
  p.active = a.active;
  p.n_active = a.n_active;
  p.pass_off = a.pass_off;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.out_f32 = static_cast<float*>(a.out_f32);
  p.N = w->N;
  p.KT = KT;
  p.NT = NT;
  p.E = w->E;
  p.P = static_cast<int>(P);
  p.ksplit = 1;
  if (!wide && a.part && a.split_slot && a.part_bytes >= moe_part_bytes(P, w->N) && moe_part_bytes(P, w->N) > 0) {
    // ranges of at least two K steps; the count is chosen on the device
    p.ksplit = KT / 2 < kMaxKSplit ? (KT / 2 > 1 ? KT / 2 : 1) : kMaxKSplit;
    p.part = static_cast<float*>(a.part);
    p.split_out = a.split_slot;
  }
  p.lo = a.lo;
  p.gate_up = w->layout == MX_LAYOUT_GATE_UP ? 1 : 0;
  p.out_mode = a.out_mode;
  if (!wide) {
    // decode sizes: the 16-row form (four weight stages a CTA), routing itself
    // from the ids before its dependency wait when the kernel before it has
    // waited for its own (act_route_kernel) or no early start is asked for
    // also above the decode sizes while the experts average at most half a
    // 16-row pass of pairs (measured on GB300, E=64 N=K=4096 top-8: A16W4 T=16
    // 89.3 -> 82.4 us, T=32 100.8 -> 98.8; MXFP8 T=16 / 32 / 64 -8 / -6.5 /
    // -3 %; A16W4 T=64, 8 pairs an expert, +46 % from the second passes)
    const bool n16 = P <= kSplitMaxPairs || 2 * P <= static_cast<long long>(w->E) * (16 >> a.lo);
    p.ids = a.ids;
    p.early = n16 && P <= kEarlyPairs && a.ids && (a.route_in_act || a.no_pdl) ? 1 : 0;
    int rc = n16 ? launch_moe_gemm<kMoeNarrow16>(a, p, xh, xl, cs, cfg) : launch_moe_gemm<kMoeNarrow>(a, p, xh, xl, cs, cfg);
    if (rc != MX_OK || p.ksplit == 1) return rc;
    // add the K ranges' partial sums (programmatic dependent of the GEMM)
    const int cols = a.out_mode == kMoeOutSwiglu ? w->N / 2 : w->N;
    const long long total = P * static_cast<long long>((cols + 3) / 4);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks_for(total, 256)), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_finish_kernel, static_cast<const float*>(p.part),
                           static_cast<const int32_t*>(a.split_slot), p.P, w->N, a.pairs, a.offsets + w->E,
                           a.out_mode, p.gate_up, static_cast<__nv_bfloat16*>(a.out), static_cast<float*>(a.out_f32));
    if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "moe finish launch: %s", cudaGetErrorString(e));
    return MX_OK;
  }
  // two 128-row tiles an item when the tiles pair up evenly (measured on
  // GB300, E=64 N=K=4096 top-8 T=4096: W4A8 775 -> 698 us; the full A16W4
  // expert, whose SiLU-and-mul and f32 epilogues the one-tile form cannot
  // hide, 2737 -> 2007 us; the plain A16W4 GEMM within 1 %)
  return NT % 2 == 0 ? launch_moe_gemm<kMoePair>(a, p, xh, xl, cs, cfg) : launch_moe_gemm<kMoeWide>(a, p, xh, xl, cs, cfg);
}

}  // namespace mx
