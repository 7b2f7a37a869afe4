// K-QUANT (per-token MXFP8 activation quantizer) and K-DEQ (MX dequant to bf16).
//
// Quantizer: rocm_native (vllm.model_executor.kernels.linear.mxfp8.rocm_native),
// _quant_mxfp8_tile.  Dequant: weights942, ocp_from_dequant (w = e4m3 value x
// 2^(code - 127)) and a16w4, dequant (fp4x2, low nibble first).
//
// Both are HBM-bound elementwise passes: each thread moves 16 bytes of bf16,
// four lanes form one 32-element MX block.

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {

namespace {

// One thread = 8 consecutive elements of a row; 4 lanes = one MX block.
// Grid-stride over 8-element groups of the [M, Kout] output (Kout >= K,
// multiple of 32).  All lanes of a warp run the same trip count, so the
// 4-lane shuffles inside mx_quant_bf16x8 always see a full warp.
__global__ void __launch_bounds__(256) quant_act_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int M, int K, int Kout,
                                                        uint8_t* __restrict__ q, int ldq,
                                                        uint8_t* __restrict__ codes, int ldc,
                                                        uint8_t pad_code, uint8_t* __restrict__ sf,
                                                        int pdl_trigger, int M_out, int* zero,
                                                        int nzero) {
  if (pdl_trigger) {
    // launched as a programmatic dependent: let the next kernel start, but
    // touch x and the outputs only once the previous kernel is complete
    pdl_launch_dependents();
    pdl_wait_prior_grid();
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
  const int groups_per_row = Kout >> 3;
  const long long total = static_cast<long long>(M_out) * groups_per_row;
  const int lane = threadIdx.x & 31;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       base < total; base += stride) {
    const long long g = base + lane;
    const bool inside = g < total;
    const int row = inside ? static_cast<int>(g / groups_per_row) : 0;
    const int k = inside ? static_cast<int>(g % groups_per_row) * 8 : 0;
    const bool valid = inside && row < M && k < K;
    const uint4 u = valid ? *reinterpret_cast<const uint4*>(x + static_cast<long long>(row) * K + k)
                          : make_uint4(0u, 0u, 0u, 0u);
    const QuantBlock8 b = mx_quant_bf16x8(u);
    if (!inside) continue;
    uint2 out = valid ? make_uint2(b.lo, b.hi) : make_uint2(0u, 0u);
    *reinterpret_cast<uint2*>(q + static_cast<long long>(row) * ldq + k) = out;
    if ((k & 31) == 0) {
      // blocks past K get pad_code; rows past M are quantized zeros (code 0)
      const uint8_t c = valid ? static_cast<uint8_t>(b.code) : (k < K ? 0 : pad_code);
      if (codes) codes[static_cast<long long>(row) * ldc + (k >> 5)] = c;
      if (sf) {
        // 512-byte atom (row tile, 128-K tile): row m, block kb at (m%32)*16 + (m/32)*4 + kb
        const int j = k >> 5;
        const int m = row & 127;
        const long long atom = static_cast<long long>(row >> 7) * (Kout >> 7) + (j >> 2);
        sf[atom * 512 + (m & 31) * 16 + (m >> 5) * 4 + (j & 3)] = c;
      }
    }
  }
}

// Dequant: one thread = 8 consecutive output elements of a row.
template <int kFmt>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ bytes,
                                                      const uint8_t* __restrict__ codes,
                                                      int block_scale, int N, int K,
                                                      __nv_bfloat16* __restrict__ out) {
  const int groups_per_row = K >> 3;
  const long long total = static_cast<long long>(N) * groups_per_row;
  const int KB = K >> 5;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g % groups_per_row) * 8;
    const int crow = block_scale ? (n >> 5) : n;
    const float s = e8m0_to_f32(codes[static_cast<long long>(crow) * KB + (k >> 5)]);
    float v[8];
    if (kFmt == MX_FMT_E4M3) {
      const uint2 u = *reinterpret_cast<const uint2*>(bytes + static_cast<long long>(n) * K + k);
      const uint32_t w[2] = {u.x, u.y};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1))));
        const float2 f = __half22float2(h);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    } else {
      const uint32_t w =
          *reinterpret_cast<const uint32_t*>(bytes + static_cast<long long>(n) * (K >> 1) + (k >> 1));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(e2m1x2_to_f16x2((w >> (8 * i)) & 0xffu));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i] * s, v[2 * i + 1] * s);
      o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(out + static_cast<long long>(n) * K + k) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// weights942, ocp_from_dequant: the e4m3 bytes behind a bf16 weight w = e4m3
// value x 2^(code - 127).  One thread = 8 consecutive elements of a row: scale
// by 2^(127 - code), round to e4m3 (nearest-even, saturating: a value beyond
// 448 fails the check below anyway), and count the values whose byte does not
// give w back (dequant rounded to bf16; -0 equals +0, a NaN never matches).
__global__ void __launch_bounds__(256) from_dequant_kernel(const __nv_bfloat16* __restrict__ w,
                                                           const uint8_t* __restrict__ codes,
                                                           int block_scale, int N, int K,
                                                           uint8_t* __restrict__ out,
                                                           unsigned long long* mismatches) {
  const int groups_per_row = K >> 3;
  const long long total = static_cast<long long>(N) * groups_per_row;
  const int KB = K >> 5;
  unsigned int bad = 0;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g % groups_per_row) * 8;
    const uint32_t c = codes[static_cast<long long>(block_scale ? (n >> 5) : n) * KB + (k >> 5)];
    const uint4 u = *reinterpret_cast<const uint4*>(w + static_cast<long long>(n) * K + k);
    const uint32_t wb[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[2] = {0x7f7f7f7fu, 0x7f7f7f7fu};
    if (c == 255u) {
      bad += 8;  // a NaN scale gives nothing back
    } else {
      // 2^(127 - c) and 2^(c - 127) as f32: exponent fields 254 - c and c, 0 -> 2^-127
      const float down = (c == 254u) ? __uint_as_float(0x00400000u) : __uint_as_float((254u - c) << 23);
      const float up = (c == 0u) ? __uint_as_float(0x00400000u) : __uint_as_float(c << 23);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = wb[i] & 0xffffu, hi = wb[i] >> 16;
        const uint32_t q = f32x2_to_e4m3x2(__uint_as_float(lo << 16) * down, __uint_as_float(hi << 16) * down);
        const float2 f = __half22float2(e4m3x2_to_f16x2(static_cast<uint16_t>(q)));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * up, f.y * up);
        const uint32_t bb = *reinterpret_cast<const uint32_t*>(&b);
        const uint32_t blo = bb & 0xffffu, bhi = bb >> 16;
        const bool ok_lo = ((blo == lo) || (((blo | lo) & 0x7fffu) == 0)) && (lo & 0x7fffu) <= 0x7f80u;
        const bool ok_hi = ((bhi == hi) || (((bhi | hi) & 0x7fffu) == 0)) && (hi & 0x7fffu) <= 0x7f80u;
        bad += (ok_lo ? 0u : 1u) + (ok_hi ? 0u : 1u);
        // bytes 2i, 2i + 1 of the 8 outputs
        const uint32_t shift = 16u * (i & 1);
        o[i >> 1] = (o[i >> 1] & ~(0xffffu << shift)) | (q << shift);
      }
    }
    *reinterpret_cast<uint2*>(out + static_cast<long long>(n) * K + k) = make_uint2(o[0], o[1]);
  }
  for (int off = 16; off > 0; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, static_cast<unsigned long long>(bad));
}

int grid_for(long long threads, int block) {
  long long g = (threads + block - 1) / block;
  DeviceInfo di;
  const int cap = (current_device_info(&di) == MX_OK) ? di.sm_count * 16 : 2048;
  if (g > cap) g = cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace

cudaError_t launch_quant_act(const void* x, int M, int K, int Kout, uint8_t* q, int ldq,
                             uint8_t* codes, int ldc, uint8_t pad_code, uint8_t* sf,
                             bool pdl_trigger, cudaStream_t stream, int M_out, int* zero,
                             int nzero) {
  if (M_out < M) M_out = M;
  const long long groups = static_cast<long long>(M_out) * (Kout / 8);
  const int block = 256;
  const int grid = grid_for(groups, block);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl_trigger ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quant_act_kernel, static_cast<const __nv_bfloat16*>(x), M, K, Kout, q, ldq,
                            codes, ldc, pad_code, sf, pdl_trigger ? 1 : 0, M_out, zero, nzero);
}

cudaError_t launch_from_dequant(const void* w, const uint8_t* codes, int block_scale, int N, int K, uint8_t* out,
                                unsigned long long* mismatches, cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / 8);
  const int grid = grid_for(groups, 256);
  from_dequant_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(w), codes, block_scale, N, K, out,
                                                mismatches);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* bytes, const uint8_t* codes, int fmt, int scale_mode,
                           int N, int K, void* out, cudaStream_t stream) {
  const long long groups = static_cast<long long>(N) * (K / 8);
  const int block = 256;
  const int grid = grid_for(groups, block);
  const int blk = scale_mode == MX_SCALE_BLOCK32X32 ? 1 : 0;
  if (fmt == MX_FMT_E4M3)
    dequant_kernel<MX_FMT_E4M3><<<grid, block, 0, stream>>>(bytes, codes, blk, N, K,
                                                             static_cast<__nv_bfloat16*>(out));
  else
    dequant_kernel<MX_FMT_E2M1><<<grid, block, 0, stream>>>(bytes, codes, blk, N, K,
                                                             static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace mx
