// Engine-peak microbenchmarks for the roofline's compute term (sm_103a).
//
// Not part of the fq C ABI: a separate library (libfq_peaks.so) that
// bench.py loads to measure, on the GPU it runs on, the throughput of each
// matrix engine the fq kernels use:
//   kind 0  mma.sync m16n8k16 f16 x f16 -> f32        (INT8 GEMM, 8-32 tokens)
//   kind 1  mma.sync m16n8k32 e4m3 x e4m3 -> f32      (legacy FP8 path)
//   kind 2  mma.sync m16n8k32 s8 x s8 -> s32          (legacy INT8 path)
//   kind 3  tcgen05.mma kind::f16, M=128 N=256 K=16, operands in shared memory
//   kind 4  tcgen05.mma kind::f8f6f4 (E4M3), M=128 N=256 K=32, operands in shared memory
//   kind 5  tcgen05.mma kind::f16, M=128 N=64 K=16 (the 64-token INT8 tile shape)
//   kind 6  tcgen05.mma kind::f8f6f4 (E4M3), M=128 N=16 K=32 (the decode einsum tile shape)
//   kind 7..10  latency (not throughput): one 128-K block of four kind::f8f6f4
//           MMAs, commit, wait - N = 16 chained / independent, N = 64 chained /
//           independent; *ops counts round trips
// Operand values are zeros: the rate of these engines does not depend on the
// data.  fq_peak_run launches one timed kernel on `stream` and writes the
// floating-point (or integer) operations it performs to *ops.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../csrc/fq_common.cuh"

namespace fqp {
using namespace fq;

constexpr int kWarps = 8;

template <int KIND>
__global__ void __launch_bounds__(kWarps * 32) mma_sync_kernel(int iters, float* sink) {
  float acc[8][4] = {};
  int iacc[8][4] = {};
  uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0, b0 = 0, b1 = 0;
  // keep operands opaque to the compiler
  if (iters < 0) a0 = a1 = a2 = a3 = b0 = b1 = 0x3c003c00u;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (KIND == 0)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(acc[c][0]), "+f"(acc[c][1]), "+f"(acc[c][2]), "+f"(acc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      else if (KIND == 1)
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(acc[c][0]), "+f"(acc[c][1]), "+f"(acc[c][2]), "+f"(acc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      else
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+r"(iacc[c][0]), "+r"(iacc[c][1]), "+r"(iacc[c][2]), "+r"(iacc[c][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int r = 0; r < 4; ++r) s += acc[c][r] + float(iacc[c][r]);
  if (s == 1.2345f) sink[threadIdx.x] = s;  // never true: keeps the work alive
}

// One thread per CTA issues `iters` MMAs (4 per 128-byte K row of the
// operands) into one TMEM accumulator, committing every 32; the CTA then
// waits (bounded) for the last commit.  KIND 3/5: kind::f16, KIND 4/6: kind::f8f6f4.
template <int KIND, int N>
__global__ void __launch_bounds__(128, 1) umma_kernel(int iters, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int A_BYTES = 128 * 128, B_BYTES = N * 128;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (A_BYTES + B_BYTES) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, N < 32 ? 32u : uint32_t(N));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid == 0) {
    const uint32_t a = smem_u32(smem), b = a + A_BYTES;
    const uint32_t idesc = umma_idesc_f16_f32(128, N);  // kind::f8f6f4 with E4M3 has the same fields
    for (int it = 0; it < iters; ++it) {
      const uint32_t koff = uint32_t(32 * (it & 3));
      const uint64_t da = umma_desc_k_sw128(a + koff), db = umma_desc_k_sw128(b + koff);
      if (KIND == 3 || KIND == 5)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(it > 0 ? 1u : 0u)
            : "memory");
      else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
            "l"(da), "l"(db), "r"(idesc), "r"(it > 0 ? 1u : 0u)
            : "memory");
    }
    umma_commit(&bar);
    if (!mbar_wait_ns(&bar, 0, 1000000000ull)) atomicOr(err, 1u);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, N < 32 ? 32u : uint32_t(N));
  }
}

// Round-trip latency of one 128-K block of kind::f8f6f4 MMAs (M=128, N, K=32
// x 4) as a pipelined consumer sees it: issue the four MMAs, commit, wait
// for the mbarrier, repeat `iters` times.  CHAIN: the four MMAs accumulate
// into one region (each depends on the previous); else each writes its own.
template <int N, bool CHAIN>
__global__ void __launch_bounds__(128, 1) umma_latency_kernel(int iters, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int A_BYTES = 128 * 128, B_BYTES = N * 128;
  constexpr uint32_t COLS = 4 * N < 32 ? 32u : uint32_t(4 * N);
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (A_BYTES + B_BYTES) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid == 0) {
    const uint32_t a = smem_u32(smem), b = a + A_BYTES;
    const uint32_t idesc = umma_idesc_f16_f32(128, N);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t da = umma_desc_k_sw128(a + 32 * j), db = umma_desc_k_sw128(b + 32 * j);
        const uint32_t d = CHAIN ? tmem : tmem + uint32_t(j * N);
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
            "l"(da), "l"(db), "r"(idesc), "r"((CHAIN && j > 0) ? 1u : 0u)
            : "memory");
      }
      umma_commit(&bar);
      if (!mbar_wait_ns(&bar, uint32_t(it & 1), 1000000000ull)) {
        atomicOr(err, 1u);
        break;
      }
      tc_fence_after();
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, COLS);
  }
}

template <int N, bool CHAIN>
static cudaError_t run_latency(int iters, int ctas, cudaStream_t s, uint32_t* err) {
  const int smem = 128 * 128 + N * 128 + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(umma_latency_kernel<N, CHAIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  umma_latency_kernel<N, CHAIN><<<ctas, 128, smem, s>>>(iters, err);
  return cudaGetLastError();
}

template <int KIND, int N>
static cudaError_t run_umma(int iters, int ctas, cudaStream_t s, uint32_t* err) {
  const int smem = 128 * 128 + N * 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(umma_kernel<KIND, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  umma_kernel<KIND, N><<<ctas, 128, smem, s>>>(iters, err);
  return cudaGetLastError();
}
}  // namespace fqp

using namespace fqp;

// Launches one engine microbenchmark (kind as listed above) with `iters`
// iterations per warp (mma.sync) or per CTA (tcgen05) over `ctas` CTAs, on
// `stream`.  *ops receives the operations performed (2 per multiply-add).
// `err` is a device word set to nonzero if a bounded wait gave up.
// Returns 0 or a cudaError_t code; -1 for an unknown kind.
extern "C" __attribute__((visibility("default"))) int fq_peak_run(int kind, int iters, int ctas, void* stream,
                                                                   double* ops, uint32_t* err, float* sink) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const double warps = double(ctas) * kWarps;
  cudaError_t e;
  switch (kind) {
    case 0:
      mma_sync_kernel<0><<<ctas, kWarps * 32, 0, s>>>(iters, sink);
      *ops = warps * iters * 8 * 2.0 * 16 * 8 * 16;
      return int(cudaGetLastError());
    case 1:
      mma_sync_kernel<1><<<ctas, kWarps * 32, 0, s>>>(iters, sink);
      *ops = warps * iters * 8 * 2.0 * 16 * 8 * 32;
      return int(cudaGetLastError());
    case 2:
      mma_sync_kernel<2><<<ctas, kWarps * 32, 0, s>>>(iters, sink);
      *ops = warps * iters * 8 * 2.0 * 16 * 8 * 32;
      return int(cudaGetLastError());
    case 3:
      e = run_umma<3, 256>(iters, ctas, s, err);
      *ops = double(ctas) * iters * 2.0 * 128 * 256 * 16;
      return int(e);
    case 4:
      e = run_umma<4, 256>(iters, ctas, s, err);
      *ops = double(ctas) * iters * 2.0 * 128 * 256 * 32;
      return int(e);
    case 5:
      e = run_umma<5, 64>(iters, ctas, s, err);
      *ops = double(ctas) * iters * 2.0 * 128 * 64 * 16;
      return int(e);
    case 6:
      e = run_umma<6, 16>(iters, ctas, s, err);
      *ops = double(ctas) * iters * 2.0 * 128 * 16 * 32;
      return int(e);
    case 7:   // round trips of a chained 4-MMA block, N = 16: *ops = round trips
      e = run_latency<16, true>(iters, ctas, s, err);
      *ops = double(iters);
      return int(e);
    case 8:   // the same with four independent accumulators
      e = run_latency<16, false>(iters, ctas, s, err);
      *ops = double(iters);
      return int(e);
    case 9:   // chained, N = 64
      e = run_latency<64, true>(iters, ctas, s, err);
      *ops = double(iters);
      return int(e);
    case 10:  // independent, N = 64
      e = run_latency<64, false>(iters, ctas, s, err);
      *ops = double(iters);
      return int(e);
    default:
      return -1;
  }
}
