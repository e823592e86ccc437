// Load-time weight repack to the K-major layout the linears stream with TMA.
//
// "DeepSeek-V4 W8A8 performance analysis", section 4: weights are cast once,
// at load time, to the layout the matmul reads best (npu_format_cast to
// FRACTAL_NZ on the pages' hardware).  Here that layout is K-major: a
// logical W[k, n] stored as w_nk[n * K + k], so one TMA box is a run of
// output channels with 128 contiguous K bytes each.  The repack is a batched
// byte transpose [B, K, N] -> [B, N, K], shared by the INT8 weights (B =
// experts or 1) and the FP8 einsum weights (B = groups, logical [G, D, N]).
//
// Untimed and off the decode path: one CTA per 64 x 64-byte tile, 16-byte
// loads and stores, the transpose done through shared memory.
#include "fq_common.cuh"

namespace fq {

constexpr int kRT = 64;           // tile edge in bytes
constexpr int kRTPad = kRT + 4;   // row pitch in shared memory (17 words: conflict-free column reads)

// src [B][K][N] bytes -> dst [B][N][K]; K % 16 == 0, N % 16 == 0.
__global__ void __launch_bounds__(256) repack_kmajor_kernel(const uint8_t* __restrict__ src, int64_t B, int64_t K,
                                                            int64_t N, uint8_t* __restrict__ dst) {
  __shared__ __align__(16) uint8_t tile[kRT * kRTPad];
  const int tid = threadIdx.x;
  const int r = tid >> 2, c16 = (tid & 3) * 16;  // row r of the tile, 16-byte chunk at column c16
  const int64_t n0 = int64_t(blockIdx.x) * kRT, k0 = int64_t(blockIdx.y) * kRT;
  for (int64_t b = blockIdx.z; b < B; b += gridDim.z) {
    const uint8_t* s = src + b * K * N;
    uint8_t* d = dst + b * K * N;
    // load rows k0 + r, columns n0 + c16 .. +15 (whole chunks: N % 16 == 0)
    if (k0 + r < K && n0 + c16 < N) {
      const uint4 v = *reinterpret_cast<const uint4*>(s + (k0 + r) * N + n0 + c16);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) tile[r * kRTPad + c16 + i] = uint8_t(w[i >> 2] >> (8 * (i & 3)));
    }
    __syncthreads();
    // store rows n0 + r of the output, K columns k0 + c16 .. +15
    if (n0 + r < N && k0 + c16 < K) {
      uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i >> 2] |= uint32_t(tile[(c16 + i) * kRTPad + r]) << (8 * (i & 3));
      *reinterpret_cast<uint4*>(d + (n0 + r) * K + k0 + c16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
}

static fq_status repack_common(const void* src, int64_t B, int64_t K, int64_t N, void* dst, int64_t k_mult,
                               int64_t n_mult, fq_stream_t stream) {
  if (B < 0 || K < 0 || N < 0 || K % k_mult || N % n_mult) return FQ_ERR_SHAPE;
  if (K > (int64_t(1) << 31) || N > (int64_t(1) << 31) || B > (int64_t(1) << 31) ||
      (K > 0 && N > 0 && B > (int64_t(1) << 46) / K / N))
    return FQ_ERR_SHAPE;
  if (B == 0 || K == 0 || N == 0) return FQ_OK;
  if (!src || !dst) return FQ_ERR_NULL;
  if (!aligned16(src) || !aligned16(dst)) return FQ_ERR_ALIGN;
  // no in-place or overlapping transpose
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t bytes = uintptr_t(B) * uintptr_t(K) * uintptr_t(N);
  if (s0 < d0 + bytes && d0 < s0 + bytes) return FQ_ERR_ARG;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int64_t gx = (N + kRT - 1) / kRT, gy = (K + kRT - 1) / kRT;
  if (gx > 0x7FFFFFFF || gy > 65535) return FQ_ERR_SHAPE;
  const unsigned gz = unsigned(B < 65535 ? B : 65535);
  // a weight producer: launched without programmatic dependent launch and
  // never triggering early, so a linear that follows starts after it finished
  repack_kmajor_kernel<<<dim3(unsigned(gx), unsigned(gy), gz), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(src), B, K, N, static_cast<uint8_t*>(dst));
  return cuda_status(cudaGetLastError());
}

}  // namespace fq

using namespace fq;

extern "C" __attribute__((visibility("default"))) fq_status fq_repack_weight_kmajor_i8(const int8_t* w_kn, int64_t B,
                                                                                      int64_t K, int64_t N,
                                                                                      int8_t* w_nk,
                                                                                      fq_stream_t stream) {
  return repack_common(w_kn, B, K, N, w_nk, 16, 16, stream);
}

extern "C" __attribute__((visibility("default"))) fq_status fq_repack_weight_kmajor_fp8(const uint8_t* w_gdn, int64_t G,
                                                                                       int64_t D, int64_t N,
                                                                                       uint8_t* w_gnd,
                                                                                       fq_stream_t stream) {
  return repack_common(w_gdn, G, D, N, w_gnd, 128, 128, stream);
}
