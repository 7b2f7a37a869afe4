// K-PACK: load-time repack of MX weights into the library's layout.
//
// Semantics kept from the pages (weights942 = vllm.models.deepseek_v41.amd.mono.
// weights942; rocm_native = vllm.model_executor.kernels.linear.mxfp8.rocm_native):
//   - K padded with zero bytes to a multiple of 128, padded blocks get code 128
//     (weights942, dense_copy);
//   - [N, K/32] row codes fold to [N/32, K/32] blocks when every 32 rows agree
//     (rocm_native, _as_block32_scale), else stay per row or are refused
//     (weights942, linear_copy);
//   - -0 nibbles become +0 and are counted (weights942, fp4_drop_negative_zero_);
//   - a K block keeps its code when bytes move inside a row (weights942,
//     fp4_lane_major).
// The byte order itself is this library's own (see include/mx.h).

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr uint8_t kPadCode = 128;
constexpr uint8_t kPadRowCode = 127;

// Packed row r of a gate / up interleaved expert -> its source row (gate rows
// first, then up rows): 8-row groups alternate gate and up.
__device__ __forceinline__ int gate_up_src_row(int r, int N) {
  const int q = r >> 4, i = r & 15;
  return i < 8 ? 8 * q + i : (N >> 1) + 8 * q + i - 8;
}

// status bit 0: a code is 255; bit 1: some row differs from its 32-row group's first row.
__global__ void check_codes_kernel(const uint8_t* __restrict__ codes, int E, int rows, int KB,
                                   int check_fold, unsigned int* status) {
  const long long total = static_cast<long long>(E) * rows * KB;
  unsigned int flags = 0;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint8_t c = codes[i];
    if (c == 255) flags |= 1u;
    if (check_fold) {
      const long long j = i % KB;
      const long long er = i / KB;  // e * rows + r
      const int r = static_cast<int>(er % rows);
      const long long first = (er - (r & 31)) * KB + j;
      if (codes[first] != c) flags |= 2u;
    }
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if ((threadIdx.x & 31) == 0 && flags) atomicOr(status, flags);
}

// E4M3 bytes [E, N, K] -> [E, N, Kp], 16 bytes a thread.
__global__ void pack_e4m3_bytes_kernel(const uint8_t* __restrict__ in, long long rows, int K,
                                       int Kp, uint8_t* __restrict__ out) {
  const int chunks = Kp >> 4;
  const long long total = rows * chunks;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / chunks;
    const int k = static_cast<int>(i % chunks) << 4;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k < K) v = *reinterpret_cast<const uint4*>(in + r * K + k);
    *reinterpret_cast<uint4*>(out + r * Kp + k) = v;
  }
}

// Code of row n, K block j, from the caller's codes ([E, N/32, KB] or [E, N, KB]).
__device__ __forceinline__ uint8_t src_row_code(const uint8_t* codes, int e, int n, int j, int N,
                                                int KB, int codes_rows) {
  const int r = (codes_rows == N) ? n : (n >> 5);
  return codes[(static_cast<long long>(e) * codes_rows + r) * KB + j];
}

// Compact codes: block mode [E, N/32, KBp] (first row of each group), row mode [E, N, KBp].
__global__ void pack_codes_kernel(const uint8_t* __restrict__ codes, int E, int N, int KB, int KBp,
                                  int codes_rows, int block_out, int gate_up, uint8_t* __restrict__ out) {
  const int orows = block_out ? (N >> 5) : N;
  const long long total = static_cast<long long>(E) * orows * KBp;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i % KBp);
    const long long er = i / KBp;
    const int r = static_cast<int>(er % orows);
    const int e = static_cast<int>(er / orows);
    const int n = block_out ? (r << 5) : (gate_up ? gate_up_src_row(r, N) : r);
    out[i] = j < KB ? src_row_code(codes, e, n, j, N, KB, codes_rows) : kPadCode;
  }
}

// SF atoms [E, ceil(N/128), Kp/128, 512]: row n = 128 rt + m, block j = 4 kt + kb
// at byte (m % 32) * 16 + (m / 32) * 4 + kb.
__global__ void pack_sf_kernel(const uint8_t* __restrict__ codes, int E, int N, int KB, int Kp,
                               int codes_rows, int gate_up, uint8_t* __restrict__ sf) {
  const int RT = (N + 127) >> 7;
  const int KT = Kp >> 7;
  const long long total = static_cast<long long>(E) * RT * KT * 512;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i & 511);
    const long long atom = i >> 9;
    const int kt = static_cast<int>(atom % KT);
    const long long ert = atom / KT;
    const int rt = static_cast<int>(ert % RT);
    const int e = static_cast<int>(ert / RT);
    const int m = (pos >> 4) + ((pos >> 2) & 3) * 32;
    const int kb = pos & 3;
    const int n = rt * 128 + m;
    const int j = kt * 4 + kb;
    uint8_t c;
    if (n >= N) c = kPadRowCode;
    else if (j >= KB) c = kPadCode;
    else c = src_row_code(codes, e, gate_up ? gate_up_src_row(n, N) : n, j, N, KB, codes_rows);
    sf[i] = c;
  }
}

__device__ __forceinline__ uint32_t drop_negative_zero_word(uint32_t w, int* count) {
  int c = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (((w >> (4 * i)) & 0xfu) == 0x8u) {
      w &= ~(0xfu << (4 * i));
      ++c;
    }
  }
  *count += c;
  return w;
}

// E2M1 bytes [E, N, K/2] -> tiles [E, NT, KT, 128, 64]: K step kt (128 values,
// 64 bytes, low nibble first) of rows 128 rt .. 128 rt + 127, one contiguous
// 8 KB block; -0 nibbles cleared, zero past K and past N, rows optionally
// gate / up interleaved.  One thread per output word.
__global__ void pack_e2m1_bytes_kernel(const uint8_t* __restrict__ in, int E, int N, int gate_up, int KH,
                                       int KT, uint8_t* __restrict__ out, unsigned long long* negz) {
  const int NT = (N + 127) >> 7;
  const long long total = static_cast<long long>(E) * NT * KT * 128 * 16;
  int count = 0;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int w = static_cast<int>(i & 15);
    const int m = static_cast<int>((i >> 4) & 127);
    const long long blk = i >> 11;  // (e, rt, kt)
    const int kt = static_cast<int>(blk % KT);
    const long long ert = blk / KT;
    const int rt = static_cast<int>(ert % NT);
    const int e = static_cast<int>(ert / NT);
    const int n = rt * 128 + m;
    const int src = kt * 64 + w * 4;
    uint32_t v = 0u;
    if (n < N && src < KH) {
      const int ns = gate_up ? gate_up_src_row(n, N) : n;
      v = drop_negative_zero_word(
          *reinterpret_cast<const uint32_t*>(in + (static_cast<long long>(e) * N + ns) * KH + src), &count);
    }
    *reinterpret_cast<uint32_t*>(out + i * 4) = v;
  }
  // warp-reduce the -0 count, one atomic a warp (integer: order-independent)
  for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xffffffffu, count, off);
  if ((threadIdx.x & 31) == 0 && count) atomicAdd(negz, static_cast<unsigned long long>(count));
}

}  // namespace

cudaError_t launch_pack_check_codes(const uint8_t* codes, int E, int rows, int KB, bool check_fold,
                                    unsigned int* status, cudaStream_t stream) {
  const long long total = static_cast<long long>(E) * rows * KB;
  check_codes_kernel<<<blocks_for(total, 256), 256, 0, stream>>>(codes, E, rows, KB,
                                                                 check_fold ? 1 : 0, status);
  return cudaGetLastError();
}

cudaError_t launch_pack_e4m3(const uint8_t* bytes, const uint8_t* codes, int E, int N, int K,
                             int Kp, int codes_rows, bool block_out, uint8_t* wq,
                             uint8_t* codes_out, uint8_t* sf, cudaStream_t stream) {
  const long long rows = static_cast<long long>(E) * N;
  pack_e4m3_bytes_kernel<<<blocks_for(rows * (Kp >> 4), 256), 256, 0, stream>>>(bytes, rows, K,
                                                                                 Kp, wq);
  const int KB = K >> 5, KBp = Kp >> 5;
  const long long ncodes = static_cast<long long>(E) * (block_out ? N / 32 : N) * KBp;
  pack_codes_kernel<<<blocks_for(ncodes, 256), 256, 0, stream>>>(codes, E, N, KB, KBp, codes_rows,
                                                                 block_out ? 1 : 0, 0, codes_out);
  const long long nsf = static_cast<long long>(E) * ((N + 127) / 128) * (Kp / 128) * 512;
  pack_sf_kernel<<<blocks_for(nsf, 256), 256, 0, stream>>>(codes, E, N, KB, Kp, codes_rows, 0, sf);
  return cudaGetLastError();
}

cudaError_t launch_act_sf_atoms(const uint8_t* codes, int M, int K, int Kp, uint8_t* sf, cudaStream_t stream) {
  const long long total = static_cast<long long>((M + 127) >> 7) * (Kp >> 7) * 512;
  pack_sf_kernel<<<blocks_for(total, 256), 256, 0, stream>>>(codes, 1, M, K >> 5, Kp, M, 0, sf);
  return cudaGetLastError();
}

cudaError_t launch_pack_e2m1(const uint8_t* bytes, const uint8_t* codes, int E, int N, int K,
                             int Kp, int codes_rows, bool gate_up, uint8_t* wq, uint8_t* codes_out,
                             uint8_t* sf, unsigned long long* negz, cudaStream_t stream) {
  const long long words = static_cast<long long>(E) * ((N + 127) / 128) * (Kp / 128) * 128 * 16;
  pack_e2m1_bytes_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(bytes, E, N, gate_up ? 1 : 0, K >> 1,
                                                                     Kp >> 7, wq, negz);
  const int KB = K >> 5, KBp = Kp >> 5;
  const long long ncodes = static_cast<long long>(E) * N * KBp;
  pack_codes_kernel<<<blocks_for(ncodes, 256), 256, 0, stream>>>(codes, E, N, KB, KBp, codes_rows,
                                                                 0, gate_up ? 1 : 0, codes_out);
  const long long nsf = static_cast<long long>(E) * ((N + 127) / 128) * (Kp / 128) * 512;
  pack_sf_kernel<<<blocks_for(nsf, 256), 256, 0, stream>>>(codes, E, N, KB, Kp, codes_rows, gate_up ? 1 : 0, sf);
  return cudaGetLastError();
}

}  // namespace mx
