// K-GEMV on the tensor cores: split-K MXFP8 decode linear for M <= 32 tokens.
//
// out = x @ w^T with the bf16 activation MXFP8-quantized per token inside the call
// and every 32-wide K block scaled by 2^(cw - 127) 2^(cx - 127)
// (rocm_native = vllm.model_executor.kernels.linear.mxfp8.rocm_native, _launch /
// apply_weights / _quant_mxfp8_tile).  At decode the layer is bound by
// streaming the weight (rocm_native, _select_cfg); the page fuses the activation
// quant into the GEMM at tiny M (apply_weights).  Here, per CTA:
//
//   * one 128-row weight tile and one K slice (the S CTAs of a cluster hold the
//     S slices of a tile); the weight boxes (128 rows x 128 bytes, 128B swizzle)
//     and their 512-byte scale atoms stream through a TMA ring from the first
//     instruction, before the previous kernel on the stream has finished;
//   * once it has, the four epilogue warps load the bf16 activation slice from
//     L2 (columns >= K read as zeros) and quantize it (same block rule as the
//     standalone quantizer) straight into the 128B-swizzled K-major layout the
//     tensor core reads, plus the activation scale atom;
//   * warp 1 issues, per K step, tcgen05.cp of both scale atoms into tensor
//     memory and four tcgen05.mma kind::mxf8f6f4.block_scale (M = 128 weight
//     rows, N = 16 or 32 token columns, K = 32): the block scales are applied
//     by the tensor core, the f32 sums stay in tensor memory.  One thread
//     issues a block-scaled MMA only about every 150 cycles (measured on
//     GB300), so when the whole slice sits in the ring (no refills) the TMA
//     thread, idle once its loads are issued, takes the odd ring stages into a
//     second accumulator; the epilogue adds the two in a fixed order;
//   * the epilogue reads the 128 x 32 accumulator (tcgen05.ld) and sends each
//     row's partial to the CTA of the cluster that owns the row, completing on
//     that CTA's mbarrier: per-thread st.async for M <= 8 over more than two
//     owners, else staged in the CTA's dead weight ring and sent with one bulk
//     copy a owner; each CTA
//     waits for the S partials of its 128 / S rows, sums them in rank order,
//     adds the bias and stores bf16.  The receive buffer has its own shared
//     memory when four CTAs per SM still fit, else it reuses the weight ring
//     once every CTA of the cluster has finished its MMAs (one cluster barrier).
// The split depends on (N, K) only, so a token's result does not depend on M.
// Every mbarrier wait is bounded.

#include "mx_common.cuh"
#include "mx_internal.h"
#include "tc_common.cuh"

namespace mx {
namespace {

constexpr int kRows = 128;                // weight rows a tile (MMA M)
constexpr int kTok = 32;                  // token columns (MMA N)
constexpr int kStepB = 128;               // K bytes a step
constexpr int kMaxRing = 6;               // weight ring depth
constexpr int kXBlocks = 2;               // MX blocks (4 x 16-byte loads each) in flight a thread
constexpr int kPushMaxM = 8;              // up to this M, partials go by per-thread st.async, above by bulk copy
constexpr int kMaxSteps = 8;              // K steps a CTA (slice)
constexpr int kThreads = 192;             // warp 0 TMA, warp 1 MMA, warps 2..5 quant + epilogue
constexpr int kWBox = kRows * kStepB;     // 16 KB
constexpr int kMaxCtasPerSm = 5;          // register budget (launch bounds)

// MMA N (token columns) for M tokens, and the quantized-activation bytes a step.
__host__ __device__ inline int mma_n(int M) { return M <= 16 ? 16 : 32; }
__host__ __device__ inline int xq_step_bytes(int M) { return mma_n(M) * kStepB; }

// MMA issuers of a CTA with `steps` K steps and a `ring`-stage weight ring:
// two (warp 1 the even stages, the TMA thread the odd ones) when the slice
// fits the ring, so that the TMA thread has no refills to make; else one.
__host__ __device__ inline int issuers_for(int steps, int ring) { return steps >= 2 && steps <= ring ? 2 : 1; }

// The slices of one call hold KT / S or KT / S + 1 steps; the tensor-memory
// layout has room for the most issuers any of them uses.
__host__ __device__ inline int issuers_layout(int KT, int S, int ring) {
  const int a = issuers_for(KT / S, ring), b = issuers_for((KT + S - 1) / S, ring);
  return a > b ? a : b;
}

// Tensor-memory columns: one accumulator (MMA N columns) a issuer of the
// layout and one scale-factor slot (SFw 4 + SFx 4 columns) a step, rounded up
// to a power of two >= 32.
__host__ __device__ inline int tmem_cols_for(int M, int KT, int S, int ring) {
  const int steps = (KT + S - 1) / S;
  const int need = issuers_layout(KT, S, ring) * mma_n(M) + steps * 8;
  int c = 32;
  while (c < need) c <<= 1;
  return c;
}
constexpr uint32_t kIdesc32 = mxf8_idesc(kRows, 32);  // 17..32 tokens
constexpr uint32_t kIdesc16 = mxf8_idesc(kRows, 16);  // 1..16 tokens: half the tensor work

struct TcGemvParams {
  const uint8_t* sfw;          // weight scale atoms [RT][KT][512]
  const __nv_bfloat16* x;      // [M, K]
  const uint8_t* xq;           // pre-quantized activation [M, K] e4m3, or null (quantize x here)
  const uint8_t* xcodes;       // its E8M0 codes [M, K/32] row-major
  const __nv_bfloat16* bias;   // [N] or null
  __nv_bfloat16* out;          // [M, N]
  int M, N, K, KT, splits, ring;
  int own_recv;                // 1: the receive buffer has its own shared memory
  int bulk;                    // 1: partials go by bulk copy, 0: by per-thread st.async
  int tmem_cols;               // tensor-memory allocation (tmem_cols_for)
};

struct Layout {
  int w, sfw, xq, sfx, recv, stage, bars, total;
};

// Shared memory.  The receive buffer of the split-K partials holds, for each
// of the S slices and each of this CTA's ceil(128 / S) rows, recv_stride(M)
// floats: M rounded up to 4, plus 4 when that is a multiple of 8, so that the
// 16-byte reads of consecutive rows fall in distinct banks.  It either has its
// own region or reuses the weight ring.
__host__ __device__ inline int recv_stride(int M) {
  const int m4 = (M + 3) & ~3;
  return (m4 & 7) == 0 ? m4 + 4 : m4;
}

__host__ __device__ inline int recv_bytes_for(int splits, int M) {
  return splits > 1 ? splits * ((kRows + splits - 1) / splits) * recv_stride(M) * 4 : 0;
}

// The CTA's own 128 x M partial is staged (by owner, in the owners' receive
// layout) in shared memory that is dead once its MMAs are done, then sent with
// one bulk copy a owner.
__host__ __device__ inline Layout layout_for(int ring, int steps, int splits, int M, bool own_recv) {
  Layout L;
  const int ring_bytes = ring * kWBox;
  const int recv_bytes = recv_bytes_for(splits, M);
  const int stage_bytes = splits > 1 ? kRows * recv_stride(M) * 4 : 0;
  L.w = 0;                                   // ring x 16 KB
  L.xq = own_recv ? ring_bytes : ((ring_bytes > recv_bytes ? ring_bytes : recv_bytes) + 1023) & ~1023;
  L.sfw = L.xq + steps * xq_step_bytes(M);   // ring x 512
  L.sfx = L.sfw + ring * 512;                // steps x 512
  const int dead_end = L.sfx + steps * 512;  // ring, xq and scale atoms: dead after the MMAs
  if (own_recv) {
    L.recv = dead_end;
    L.stage = 0;
    L.bars = L.recv + recv_bytes;
    if (stage_bytes > dead_end) {            // (never at the decode shapes) stage past recv
      L.stage = L.bars;
      L.bars += stage_bytes;
    }
  } else {
    L.recv = 0;
    L.stage = (recv_bytes + 15) & ~15;
    L.bars = dead_end > L.stage + stage_bytes ? dead_end : L.stage + stage_bytes;
  }
  L.total = L.bars + 256;
  return L;
}

// Two weight stages a CTA: with three or four CTAs per SM that keeps 96-128 KB
// of weight requests in flight on every SM.
constexpr int kDefaultRing = 2;
constexpr int kMaxAutoRing = 4;
constexpr int kWholeSlice = 5;            // K steps a CTA up to which a whole slice may sit in the ring
constexpr int kLongSlice = 8;             // K steps a CTA from which M > 16 takes kMaxAutoRing stages

__global__ void __launch_bounds__(kThreads, kMaxCtasPerSm) gemv_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const TcGemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = p.splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = blockIdx.y;
  const int base = p.KT / p.splits, rem = p.KT % p.splits;
  const int st0 = split * base + (split < rem ? split : rem);
  const int ns = base + (split < rem ? 1 : 0);
  const int ring = p.ring;
  const Layout L = layout_for(ring, (p.KT + p.splits - 1) / p.splits, p.splits, p.M, p.own_recv != 0);
  const int xqb = xq_step_bytes(p.M);                          // quantized activation a step
  const int nN = mma_n(p.M);
  const int n_iss = issuers_for(ns, ring);                                 // this CTA's MMA issuers
  const uint32_t sf_base =                                                  // scale-factor slots after the accumulators
      static_cast<uint32_t>(issuers_layout(p.KT, p.splits, ring) * nN);
  const int S = p.splits;
  const int rows_per = (kRows + S - 1) / S;        // rows each CTA of the cluster owns
  const int Mp = recv_stride(p.M);                 // receive-buffer floats a (slice, row)
  const int own_lo = split * rows_per;
  const int own_hi = own_lo + rows_per < kRows ? own_lo + rows_per : kRows;
  const int own_rows = own_hi > own_lo ? own_hi - own_lo : 0;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* wempty = wfull + kMaxRing;
  uint64_t* xready = wempty + kMaxRing;  // [kMaxSteps]: step i's quantized activation written (128 arrivals)
  uint64_t* accfull = xready + kMaxSteps;
  uint64_t* redbar = accfull + 1;        // this CTA's rows: all S partials received
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(redbar + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxRing; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < kMaxSteps; ++s) mbar_init(&xready[s], 128);
    mbar_init(accfull, static_cast<uint32_t>(n_iss));  // one commit a issuer
    mbar_init(redbar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    fence_proxy_async_smem();
    // armed now; completes once the S partials of the owned rows have landed
    // bulk copies move whole receive rows (Mp floats); per-thread pushes M rounded up to 4
    if (S > 1)
      mbar_arrive_expect_tx(redbar, static_cast<uint32_t>(S * own_rows * (p.bulk ? Mp : (p.M + 3) & ~3) * 4));
  }
  if (warp == 1) tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The next kernel may start streaming its own weights.  Triggered only
  // once this CTA holds its tensor memory: a dependent grid's CTAs then never
  // take columns that a CTA of this grid still waits for.
  pdl_launch_dependents();
  // with its own receive buffer a CTA may be pushed to as soon as its
  // barriers exist: the cluster barrier's arrive goes here, its wait just
  // before the first push (off the critical path)
  if (S > 1 && p.own_recv) cluster_arrive_release();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&wmap);
    const uint64_t pol_w = policy_evict_first();
    // the weight is immutable: it streams while earlier kernels finish
    const int first = ns < ring ? ns : ring;
    for (int i = 0; i < first; ++i) {
      mbar_arrive_expect_tx(&wfull[i], kWBox + 512);
      tma_load_2d(smem + L.w + i * kWBox, &wmap, &wfull[i], (st0 + i) * kStepB, tile * kRows, pol_w);
      bulk_load(smem + L.sfw + i * 512, p.sfw + (static_cast<long long>(tile) * p.KT + st0 + i) * 512, 512, &wfull[i]);
    }
    for (int i = first; i < ns && !*abort_flag; ++i) {
      const int stage = i % ring;
      if (!mbar_wait(&wempty[stage], (static_cast<uint32_t>(i / ring) & 1u) ^ 1u)) { *abort_flag = 1u; break; }
      mbar_arrive_expect_tx(&wfull[stage], kWBox + 512);
      tma_load_2d(smem + L.w + stage * kWBox, &wmap, &wfull[stage], (st0 + i) * kStepB, tile * kRows, pol_w);
      bulk_load(smem + L.sfw + stage * 512, p.sfw + (static_cast<long long>(tile) * p.KT + st0 + i) * 512, 512,
                &wfull[stage]);
    }
    if (n_iss == 2) {
      // ---------------------------------------------------- second MMA issuer
      // every load is issued (the slice fits the ring): the odd stages' scale
      // atoms, then, once the activation is ready, their MMAs into the second
      // accumulator (columns nN .. 2 nN - 1)
      bool ok = true;
      for (int i = 1; i < ns && ok; i += 2) {
        if (!mbar_wait(&wfull[i], 0u)) { *abort_flag = 1u; ok = false; break; }
        tc_fence_after();
        tc_cp_sf(tmem + sf_base + static_cast<uint32_t>(i * 8), sf_desc(smem_u32(smem + L.sfw + i * 512)));
      }
      const uint32_t idesc_n = p.M <= 16 ? kIdesc16 : kIdesc32;
      // up to 8 tokens every step is signalled at once: one wait, on the last
      const bool per_step = p.M > 8;
      if (ok && !per_step && !mbar_wait(&xready[ns - 1], 0)) { *abort_flag = 1u; ok = false; }
      for (int i = 1; i < ns && ok; i += 2) {
        if (per_step && !mbar_wait(&xready[i], 0)) { *abort_flag = 1u; ok = false; break; }
        tc_fence_after();
        const uint32_t sf = tmem + sf_base + static_cast<uint32_t>(i * 8);
        tc_cp_sf(sf + 4, sf_desc(smem_u32(smem + L.sfx + i * 512)));
        const uint64_t adesc = sw128_desc(smem_u32(smem + L.w + i * kWBox));
        const uint64_t bdesc = sw128_desc(smem_u32(smem + L.xq + i * xqb));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t idesc = idesc_n | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
          tc_mma_mxf8(tmem + static_cast<uint32_t>(nN), adesc + 2 * k, bdesc + 2 * k, idesc, sf, sf + 4,
                      (i > 1 || k > 0) ? 1u : 0u);
        }
      }
      tc_commit(accfull);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // a scale-factor slot per step (SFw in its first 4 columns, SFx in the
    // next 4): no step overwrites columns an earlier, possibly still running
    // MMA reads.  The weight scales of the stages already in flight go to
    // tensor memory before the activation is ready.
    bool ok = true;
    const int pre = ns < ring ? ns : ring;
    const uint32_t idesc_n = p.M <= 16 ? kIdesc16 : kIdesc32;
    const bool per_step = p.M > 8;  // else every step is signalled at once: one wait, on the last
    for (int i = 0; i < pre && ok; i += n_iss) {
      if (!mbar_wait(&wfull[i], 0u)) { *abort_flag = 1u; ok = false; break; }
      tc_fence_after();
      tc_cp_sf(tmem + sf_base + static_cast<uint32_t>(i * 8), sf_desc(smem_u32(smem + L.sfw + i * 512)));
    }
    for (int i = 0; i < ns && ok; i += n_iss) {
      const int stage = i % ring;
      const uint32_t sf = tmem + sf_base + static_cast<uint32_t>(i * 8);
      if (i >= pre) {
        if (!mbar_wait(&wfull[stage], static_cast<uint32_t>(i / ring) & 1u)) { *abort_flag = 1u; ok = false; break; }
        tc_fence_after();
        tc_cp_sf(sf, sf_desc(smem_u32(smem + L.sfw + stage * 512)));
      }
      // step i's activation (above 8 tokens the quantizing warps signal each
      // step as it is written, so the MMAs of the first steps overlap the
      // quantization of the later ones)
      if ((per_step || i == 0) && !mbar_wait(&xready[per_step ? i : ns - 1], 0)) {
        *abort_flag = 1u;
        ok = false;
        break;
      }
      tc_fence_after();
      tc_cp_sf(sf + 4, sf_desc(smem_u32(smem + L.sfx + i * 512)));
      const uint64_t adesc = sw128_desc(smem_u32(smem + L.w + stage * kWBox));
      const uint64_t bdesc = sw128_desc(smem_u32(smem + L.xq + i * xqb));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t idesc = idesc_n | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
        tc_mma_mxf8(tmem, adesc + 2 * k, bdesc + 2 * k, idesc, sf, sf + 4, (i | k) != 0 ? 1u : 0u);  // i = 0 first
      }
      if (i + ring < ns) tc_commit(&wempty[stage]);  // the producer refills this stage
    }
    tc_commit(accfull);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ quantize the slice
    const int et = threadIdx.x - 64;  // 0..127
    // the activation may be written by the previous kernel on the stream
    pdl_wait_prior_grid();
    // Only the M real token rows are quantized: rows >= M feed only output
    // columns that are never stored (every column of the MMA is independent).
    // row = (step, token) of the slice; row / M by a multiply-shift, exact for
    // rows < 2^16 / M (rows <= 8 x 32)
    const int mrows = p.M;
    const int items = ns * mrows * 16;
    const int mmul = (65536 + mrows - 1) / mrows;
    if (p.xq != nullptr) {
      // the activation arrives quantized: copy its bytes and codes into place
      for (int it = et; it < items; it += 128) {
        const int row = it >> 4, step = (row * mmul) >> 16, t = row - step * mrows, g8 = it & 15;
        const int col = (st0 + step) * kStepB + g8 * 8;
        uint2 v = make_uint2(0u, 0u);
        uint8_t code = 0;
        if (col < p.K) {
          v = __ldcg(reinterpret_cast<const uint2*>(p.xq + static_cast<long long>(t) * p.K + col));
          code = p.xcodes[static_cast<long long>(t) * (p.K >> 5) + (col >> 5)];
        }
        const int c = g8 >> 1;  // 16-byte chunk of the 128-byte row, 128B swizzle
        *reinterpret_cast<uint2*>(smem + L.xq + step * xqb + t * kStepB + ((c ^ (t & 7)) << 4) + (g8 & 1) * 8) = v;
        if ((g8 & 3) == 0) smem[L.sfx + step * 512 + t * 16 + (g8 >> 2)] = code;
      }
    }
    // bf16 activation: one whole 32-element MX block a thread (item = (step,
    // token, block)), kXBlocks blocks in flight a thread.  Items are
    // step-major, so above 8 tokens, once a thread moves past a step it
    // arrives on that step's barrier: the MMAs of a step start as soon as its
    // 128 threads are past it (measured on GB300, us a call at M = 16 / 32:
    // N=7168 K=8192 15.31 / 24.64 -> 14.29 / 21.80, N=7168 K=2048 6.10 / 7.71
    // -> 6.04 / 7.40).  Up to 8 tokens there is too little to overlap and
    // every step is signalled at the end (signalling as it goes cost 1-3 %).
    const int blocks = ns * mrows * 4;
    const bool per_step = mrows > 8;
    int arrived = 0;  // steps below this one are signalled by this thread
    for (int b0 = et; b0 < blocks && p.xq == nullptr; b0 += 128 * kXBlocks) {
      uint4 u[kXBlocks][4];
#pragma unroll
      for (int j = 0; j < kXBlocks; ++j) {
        const int ib = b0 + j * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) u[j][q] = make_uint4(0u, 0u, 0u, 0u);
        if (ib < blocks) {
          const int row = ib >> 2, step = (row * mmul) >> 16, t = row - step * mrows, kb = ib & 3;
          const int col = (st0 + step) * kStepB + kb * 32;
          if (col < p.K) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<long long>(t) * p.K + col);
#pragma unroll
            for (int q = 0; q < 4; ++q) u[j][q] = __ldcg(src + q);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kXBlocks; ++j) {
        const int ib = b0 + j * 128;
        if (ib >= blocks) break;
        const int row = ib >> 2, step = (row * mmul) >> 16, t = row - step * mrows, kb = ib & 3;
        uint4 q8[2];
        const uint32_t code = mx_quant_bf16x32(u[j], q8);
        // the block's 32 bytes are 16-byte chunks 2 kb and 2 kb + 1 of the
        // 128-byte row, 128B swizzle
        uint8_t* rowp = smem + L.xq + step * xqb + t * kStepB;
        *reinterpret_cast<uint4*>(rowp + (((2 * kb) ^ (t & 7)) << 4)) = q8[0];
        *reinterpret_cast<uint4*>(rowp + (((2 * kb + 1) ^ (t & 7)) << 4)) = q8[1];
        smem[L.sfx + step * 512 + t * 16 + kb] = static_cast<uint8_t>(code);
      }
      // this thread's later items are all in step `upto` or later
      const int nb = b0 + 128 * kXBlocks;
      const int upto = nb < blocks ? (((nb >> 2) * mmul) >> 16) : ns;
      if (per_step && upto > arrived) {
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
        for (; arrived < upto; ++arrived) mbar_arrive(&xready[arrived]);
      }
    }
    if (arrived < ns) {
      fence_proxy_async_smem();
      for (; arrived < ns; ++arrived) mbar_arrive(&xready[arrived]);
    }

    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, r = q * 32 + lane;
    const int n = tile * kRows + r;
    uint32_t acc[32];
    const bool done = mbar_wait(accfull, 0);
    // every MMA of this CTA has completed, so its weight ring is dead: peers
    // may push partials over it
    if (S > 1 && !p.own_recv) cluster_arrive_release();
    if (done) {
      tc_fence_after();
      // the accumulator(s), 16 columns at a time: the first, plus the second
      // issuer's in a fixed order (the result does not depend on M)
      const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
#pragma unroll
      for (int c0 = 0; c0 < kTok; c0 += 16) {
        if (c0 < p.M) {
          uint32_t t2[16];
          tmem_ld16_async(tmem + lanes + static_cast<uint32_t>(c0), acc + c0);
          if (n_iss == 2) tmem_ld16_async(tmem + lanes + static_cast<uint32_t>(nN + c0), t2);
          tmem_wait_ld();
          if (n_iss == 2) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              acc[c0 + j] = __float_as_uint(__uint_as_float(acc[c0 + j]) + __uint_as_float(t2[j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c0 + j] = 0u;
        }
      }
    } else {
      *abort_flag = 1u;
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[t] = 0u;
    }
    tc_fence_before();
    if (S == 1) {
      if (n < p.N) {
        const float b = p.bias ? __bfloat162float(p.bias[n]) : 0.0f;
#pragma unroll
        for (int t = 0; t < kTok; ++t)
          if (t < p.M) p.out[static_cast<long long>(t) * p.N + n] = __float2bfloat16_rn(__uint_as_float(acc[t]) + b);
      }
    } else if (!p.bulk) {
      // few tokens: push this row's partial straight to the CTA that owns it
      // (st.async onto the owner's mbarrier)
      cluster_wait_acquire();  // the owners' barriers (and, if shared, buffers) are ready
      const int owner = r / rows_per;
      const int rr = r - owner * rows_per;
      const uint32_t dst = map_shared_rank(smem_u32(smem + L.recv), static_cast<uint32_t>(owner)) +
                           static_cast<uint32_t>((split * rows_per + rr) * Mp * 4);
      const uint32_t bar = map_shared_rank(smem_u32(redbar), static_cast<uint32_t>(owner));
#pragma unroll
      for (int t = 0; t < kTok; t += 4)
        if (t < p.M)
          st_async_v4_f32(dst + static_cast<uint32_t>(t * 4), __uint_as_float(acc[t]), __uint_as_float(acc[t + 1]),
                          __uint_as_float(acc[t + 2]), __uint_as_float(acc[t + 3]), bar);
    } else {
      // stage this row's partial where its owner keeps slice `split`:
      // stage[owner][row - owner * rows_per][t], then one bulk copy a owner
      const int owner = r / rows_per;
      const int rr = r - owner * rows_per;
      float* stage = reinterpret_cast<float*>(smem + L.stage) + (owner * rows_per + rr) * Mp;
#pragma unroll
      for (int t = 0; t < kTok; t += 4)
        if (t < p.M)
          *reinterpret_cast<float4*>(stage + t) = make_float4(__uint_as_float(acc[t]), __uint_as_float(acc[t + 1]),
                                                              __uint_as_float(acc[t + 2]), __uint_as_float(acc[t + 3]));
      fence_proxy_async_smem();   // the staged partials -> visible to the bulk copies
      named_barrier(1, 128);      // the 4 epilogue warps
      cluster_wait_acquire();     // the owners' barriers (and, if shared, buffers) are ready
      if (threadIdx.x == 64) {
        for (int o = 0; o < S; ++o) {
          const int lo = o * rows_per;
          const int rows = (lo + rows_per < kRows ? rows_per : kRows - lo);
          if (rows <= 0) continue;
          const uint32_t src = smem_u32(smem + L.stage) + static_cast<uint32_t>(lo * Mp * 4);
          const uint32_t dst = map_shared_rank(smem_u32(smem + L.recv), static_cast<uint32_t>(o)) +
                               static_cast<uint32_t>(split * rows_per * Mp * 4);
          bulk_copy_to_peer(dst, src, static_cast<uint32_t>(rows * Mp * 4),
                            map_shared_rank(smem_u32(redbar), static_cast<uint32_t>(o)));
        }
        bulk_commit();
      }
    }
  }

  if (S > 1) {
    if (warp < 2) {
      // the TMA and MMA warps take part in the cluster barrier too
      if (!p.own_recv) cluster_arrive_release();
      cluster_wait_acquire();
    }
    // the S partials of this CTA's rows have landed; sum them in rank order
    if (!mbar_wait_cluster(redbar, 0)) *abort_flag = 1u;
    // item = (4-token group, owned row): consecutive threads take consecutive
    // rows, so each 16-byte read hits its own banks and the stores of a token
    // are contiguous
    const float* recv = reinterpret_cast<const float*>(smem + L.recv);
    const int groups = (p.M + 3) / 4;
    for (int idx = threadIdx.x; idx < own_rows * groups; idx += kThreads) {
      const int g4 = idx / own_rows, rr = idx % own_rows;
      const int n = tile * kRows + own_lo + rr;
      if (n >= p.N) continue;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int s = 0; s < S; ++s) {
        const float4 u = *reinterpret_cast<const float4*>(recv + (s * rows_per + rr) * Mp + 4 * g4);
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
      }
      const float b = p.bias ? __bfloat162float(p.bias[n]) : 0.0f;
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = 4 * g4 + j;
        if (t < p.M) p.out[static_cast<long long>(t) * p.N + n] = __float2bfloat16_rn(vv[j] + b);
      }
    }
  }
  if (S > 1 && p.bulk && threadIdx.x == 64) bulk_wait_read_all();  // the staged partials were read
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

}  // namespace

unsigned int take_error_flags_gemv_tc() { return take_tu_error_flags(); }

// Splits along K.  First choice: the largest power of two (<= 8) giving at
// most 1.5 CTAs per SM with at most kWholeSlice K steps a CTA, whose whole
// slice then sits in the weight ring: two consecutive calls' grids stay
// resident together (measured on GB300, N=7168, us a call at M = 1 / 4 / 16
// / 32: K=2048 4.87 / 4.93 / 6.07 / 8.31 -> 4.99 / 5.08 / 5.93 / 7.68 with 4
// splits instead of 8, K=2080 5.73 / 6.01 / 7.64 / 10.01 -> 5.32 / 5.60 /
// 6.94 / 9.09).  Else the largest power of two giving at most three
// CTAs per SM, so the grid runs as one wave with short slices requested at
// once; more splits only when a slice would exceed kMaxSteps.  Depends on
// (N, K) and the SM count, never on M.
static int gemv_tc_whole_splits(int RT, int KT, int sms) {
  int best = 0;
  for (int S = 1; S <= 8 && S <= KT; S *= 2)  // every slice at least one K step
    if (2 * RT * S <= 3 * sms && (KT + S - 1) / S <= kWholeSlice) best = S;
  return best;
}

int gemv_tc_splits(int N, int Kp, int sms, int force) {
  const int RT = (N + kRows - 1) / kRows, KT = Kp / kStepB;
  if (force > 0) return force;
  const int whole = gemv_tc_whole_splits(RT, KT, sms);
  if (whole > 0) return whole;
  int S = 1;
  while (S < 8 && 2 * S <= KT && RT * 2 * S <= 3 * sms) S *= 2;
  while ((KT + S - 1) / S > kMaxSteps && S < 8) ++S;
  return S;
}

int launch_gemv_tc(const TcGemvArgs& a, cudaStream_t stream) {
  const mx_packed_weight* w = a.w;
  DeviceInfo di;
  if (current_device_info(&di) != MX_OK) return MX_ERR_CUDA;
  TcGemvParams p = {};
  p.sfw = w->sf;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.xq = a.xq;
  p.xcodes = a.xcodes;
  p.bias = static_cast<const __nv_bfloat16*>(a.bias);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = a.M;
  p.N = w->N;
  p.K = w->K;
  p.KT = w->Kp / kStepB;
  p.splits = gemv_tc_splits(w->N, w->Kp, di.sm_count, a.force_splits);
  if (p.splits < 1 || p.splits > 8) return set_error(MX_ERR_ARG, "gemv: split count %d outside 1..8", p.splits);
  if (p.splits > 8) return set_error(MX_ERR_UNSUPPORTED, "gemv: K = %d is too long for the decode GEMV", w->K);
  const int steps = (p.KT + p.splits - 1) / p.splits;
  // Shared memory and CTAs per SM (measured on GB300): its own receive buffer
  // as long as that keeps min(4, what sharing the weight ring would keep)
  // CTAs on an SM; five CTAs per SM up to 16 tokens (N = 16 MMAs), four above
  // (the two 32-column accumulators then take 128 tensor-memory columns, and
  // the activation quantization of five co-resident CTAs costs more than the
  // extra overlap gains).  Never so little shared memory that more CTAs
  // would be resident than the tensor memory holds (their tcgen05.alloc
  // would wait on CTAs that may themselves wait on cluster peers) or than the
  // register budget allows.
  const int smem_sm = static_cast<int>(di.smem_per_sm), reserved = static_cast<int>(di.smem_reserved_per_block);
  auto per_sm = [&](int bytes) { return smem_sm / (bytes + reserved); };
  auto smem_for = [&](int ring, int* own) {
    const int alias = layout_for(ring, steps, p.splits, a.M, false).total + 1024;
    const int sep = layout_for(ring, steps, p.splits, a.M, true).total + 1024;
    const int keep = per_sm(alias) < 4 ? per_sm(alias) : 4;
    *own = p.splits > 1 && (a.force_recv ? a.force_recv == 2 : per_sm(sep) >= keep) ? 1 : 0;
    const int t = *own ? sep : alias;
    const int tmem_cap = 512 / tmem_cols_for(a.M, p.KT, p.splits, p.ring);
    int cap = a.force_cap > 0 ? a.force_cap : (a.M <= 16 ? kMaxCtasPerSm : 4);
    if (cap > kMaxCtasPerSm) cap = kMaxCtasPerSm;
    if (cap > tmem_cap) cap = tmem_cap;
    const int floor_bytes = smem_sm / (cap + 1) - reserved + 16;  // cap + 1 CTAs never fit
    return t > floor_bytes ? t : floor_bytes;
  };
  static int smem_set[64];
  // Weight ring depth: the whole slice when the split was chosen for that;
  // else two stages while the grid has more than two CTAs an SM (3-5 stay
  // resident; N=7168 K=8192 at M = 1 / 16: 16.7 / 20.4 -> 12.9 / 15.3 us with
  // two instead of four), four with at most two (N=2048 K=7168 at M = 1 / 32:
  // 7.45 / 12.25 -> 5.96 / 10.90 us; N=4096 K=7168, 224 CTAs: 8.99 / 14.13 ->
  // 7.74 / 11.83 us with 8 slices) or, above
  // 16 tokens (four CTAs an SM at most), for slices of kLongSlice steps and
  // more (N=7168 K=8192 M = 32: 26.7 with two, 24.5 us with four).  Measured
  // on GB300; the depth never changes a result, so it may follow M.
  const int RTn = (w->N + kRows - 1) / kRows;
  if (a.force_ring > 0) {
    const int r = a.force_ring < kMaxRing ? a.force_ring : kMaxRing;
    p.ring = steps < r ? steps : r;
  } else if (!a.force_splits && p.splits == gemv_tc_whole_splits(RTn, p.KT, di.sm_count)) {
    p.ring = steps;
  } else {
    const int grid = RTn * p.splits;
    int r = grid <= 2 * di.sm_count || (a.M > 16 && steps >= kLongSlice) ? kMaxAutoRing : kDefaultRing;
    if (r == kDefaultRing && a.M <= 16 && p.KT / p.splits > 3) {
      // a third stage while the grid keeps at least 15 % of the CTA slots
      // spare for the next call (N=24576 K=1536, 384 CTAs, at M = 1 / 16:
      // 9.48 / 13.77 -> 8.42 / 11.17 us; N=7168 K=8192, 448 CTAs: slower).
      // Only when every slice is longer than 3 steps: a slice that fits the
      // ring whole takes a second MMA issuer and accumulator (issuers_for),
      // which would change the summation order between M = 16 and 17.
      p.ring = 3;
      int own3 = 0;
      if (per_sm(smem_for(3, &own3)) * di.sm_count * 20 >= grid * 23) r = 3;
    }
    p.ring = steps < r ? steps : r;
  }
  const int smem = smem_for(p.ring, &p.own_recv);
  p.tmem_cols = tmem_cols_for(a.M, p.KT, p.splits, p.ring);
  // per-thread pushes win only for few tokens spread over many owners
  p.bulk = (a.M > kPushMaxM || p.splits <= 2 || a.force_bulk) ? 1 : 0;
  if (steps > kMaxSteps || static_cast<size_t>(smem) > di.max_smem_optin)
    return set_error(MX_ERR_UNSUPPORTED, "gemv: %d K steps a CTA (%d bytes of shared memory) is too many", steps, smem);
  if (reinterpret_cast<uintptr_t>(a.xq ? static_cast<const void*>(a.xq) : a.x) % 16 != 0)
    return set_error(MX_ERR_ALIGN, "gemv: the activation needs 16-byte alignment");
  CUtensorMap wmap;
  const int rc = encode_tensor_map_2d(&wmap, w->bytes, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->Kp, w->N, w->Kp, kStepB,
                                      kRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != MX_OK) return rc;
  if (raise_smem_limit(reinterpret_cast<const void*>(gemv_tc_kernel), smem, di, smem_set) != MX_OK) return MX_ERR_CUDA;
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, (w->N + kRows - 1) / kRows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel, wmap, p);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "gemv_tc launch: %s", cudaGetErrorString(e));
  return MX_OK;
}

}  // namespace mx
