// Quantization kernels of the decode path (sm_103a).
//
//  * dynamic_quant_int8      per-token INT8 quant  ("DeepSeek-V4 W8A8
//                            performance analysis", sections 1-2)
//  * swiglu_quant_int8       SwiGLU + per-token INT8 re-quant ("Reshaping LLM
//                            inference dataflow: DeepSeek V4 950", section 2.3)
//  * moe_gather_rows_i8      expert-order gather of quantized rows (same page,
//                            section 3.2)
//  * quant_fp8_group_*       FP8 E4M3 per-128 group quant writing packed UE8M0
//                            scales ("SGLang PR #34277 digest", implementation
//                            breakdown items 1-2, key source snippets)
//  * fq_pack_scales_ue8m0    the separate fp32 -> packed conversion that the PR
//                            removed (motivation section), kept as the A/B control
//  * fq_quantize_weight_fp8_block   load-time fp8 weight prep
//
// All are HBM-streaming kernels: 16-byte coalesced loads and stores,
// warp-shuffle reductions, grids sized to a multiple of the SM count.
#include <cstdlib>
#include <cstring>

#include <mutex>

#include "fq_common.cuh"

namespace fq {

// Block-wide max over blockDim.x threads (multiple of 32); `red` holds 32 floats.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = (lane < nw) ? red[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
  __syncthreads();  // `red` is reused by the next row
  return r;
}

// ---------------------------------------------------------------- a1: per-token INT8

// One CTA per row (grid-stride over rows).  Each thread keeps up to VPT
// 16-byte vectors (8 bf16) of the row in registers between the absmax pass
// and the quant pass; longer rows re-read the remainder (L2-resident).
// trigger: let the next kernel launch early.  Only for outputs that are
// activations: a dependent may read its weight operand before its own wait,
// so a call whose output could be that weight (the public entry point: a
// per-row quant of W is the per-channel weight quant) lets the next kernel
// start only once it has finished.
template <int VPT, int MAXT = 256>
__global__ void __launch_bounds__(MAXT) dynamic_quant_int8_kernel(const uint4* __restrict__ x, int64_t M,
                                                                  int64_t K8, uint2* __restrict__ q,
                                                                  float* __restrict__ s, int trigger) {
  __shared__ float red[32];
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* xr = x + row * K8;
    uint4 v[VPT];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      if (idx < K8) {
        v[i] = ld_stream(xr + idx);
        amax = fmaxf(amax, absmax8_bf16(v[i]));
      }
    }
    for (int64_t idx = tid + int64_t(VPT) * nt; idx < K8; idx += nt) amax = fmaxf(amax, absmax8_bf16(xr[idx]));
    amax = block_max(amax, red);
    const float sc = __fdiv_rn(amax, 127.0f);
    const float inv = __frcp_rn(sc);
    if (tid == 0) s[row] = sc;
    uint2* qr = q + row * K8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      if (idx < K8) {
        float f[8];
        unpack8(v[i], f);
        qr[idx] = quant8_i8(f, sc, inv);
      }
    }
    for (int64_t idx = tid + int64_t(VPT) * nt; idx < K8; idx += nt) {
      float f[8];
      unpack8(xr[idx], f);
      qr[idx] = quant8_i8(f, sc, inv);
    }
  }
}

// Many rows (M above the SM count): one CTA per row as above, grid-stride,
// with the next row's loads issued before the current row is reduced and
// stored, so each CTA keeps two rows of loads in flight; the block reduction
// scratch alternates between two buffers, which saves its trailing barrier.
template <int VPT, int MAXT, int MINB, int AH = 1>
__global__ void __launch_bounds__(MAXT, MINB) quant_int8_stream_kernel(const uint4* __restrict__ x, int64_t M, int64_t K8,
                                                                 uint2* __restrict__ q, float* __restrict__ s,
                                                                 int trigger) {
  __shared__ float red[2][32];
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
  int64_t row = blockIdx.x;
  if (row >= M) return;
  // rows row, row + grid, ..., row + AH * grid in flight (pre[0] = the current row;
  // 2 or 3 rows ahead measured no faster than 1 at M=16384, K=4096 on GB300)
  uint4 pre[AH + 1][VPT];
#pragma unroll
  for (int a = 0; a < AH; ++a) {
    const int64_t rr = row + int64_t(a) * gridDim.x;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      pre[a][i] = (rr < M && idx < K8) ? ld_stream(x + rr * K8 + idx) : make_uint4(0, 0, 0, 0);
    }
  }
  uint4 (&cur)[VPT] = pre[0];
  for (int par = 0; row < M; row += gridDim.x, par ^= 1) {
    const int64_t next = row + int64_t(AH) * gridDim.x;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      pre[AH][i] = (next < M && idx < K8) ? ld_stream(x + next * K8 + idx) : make_uint4(0, 0, 0, 0);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) amax = fmaxf(amax, absmax8_bf16(cur[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) red[par][warp] = amax;
    __syncthreads();
    float r = lane < nw ? red[par][lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
    const float sc = __fdiv_rn(r, 127.0f);
    const float inv = __frcp_rn(sc);
    if (tid == 0) s[row] = sc;
    uint2* qr = q + row * K8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      if (idx < K8) {
        float f[8];
        unpack8(cur[i], f);
        qr[idx] = quant8_i8(f, sc, inv);
      }
#pragma unroll
      for (int a = 0; a < AH; ++a) pre[a][i] = pre[a + 1][i];
    }
  }
}

// Many rows, rows of up to 8192 elements: each row is staged into a ring of
// R shared-memory slots by a 1-D bulk copy (the TMA engine) that one thread
// issues R rows ahead, so a CTA keeps R rows of loads in flight (3 CTAs of a
// 64 KB ring per SM: ~190 KB, enough to cover loaded HBM latency) while its
// threads reduce and quantize the oldest.  Rows of this CTA: blockIdx.x +
// i * gridDim.x.  Every thread waits (bounded) on the slot's barrier; a
// barrier that also votes on those waits keeps all threads in step if one
// gives up, and the copies still in flight are then drained before exit.
constexpr int kRingMax = 16;
template <int VPT>
__global__ void __launch_bounds__(256, 3) quant_int8_ring_kernel(const uint4* __restrict__ x, int64_t M, int64_t K8,
                                                                 uint2* __restrict__ q, float* __restrict__ s,
                                                                 int trigger, int R, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kRingMax];
  __shared__ float red[2][8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const uint32_t row_bytes = uint32_t(K8) * 16u;
  if (tid == 0) {
    for (int i = 0; i < R; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  const int64_t G = gridDim.x;
  const int64_t nrows = M > int64_t(blockIdx.x) ? (M - 1 - blockIdx.x) / G + 1 : 0;
  if (tid == 0) {
    for (int64_t i = 0; i < nrows && i < R; ++i) {
      mbar_arrive_expect_tx(&full[i], row_bytes);
      bulk_load(ring + i * row_bytes, x + (blockIdx.x + i * G) * K8, row_bytes, &full[i]);
    }
  }
  for (int64_t i = 0; i < nrows; ++i) {
    const int slot = int(i % R);
    const int64_t row = blockIdx.x + i * G;
    const bool ok = mbar_wait(&full[slot], uint32_t((i / R) & 1));
    const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(slot) * row_bytes);
    uint4 v[VPT];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t idx = tid + 256 * j;
      v[j] = (ok && idx < K8) ? src[idx] : make_uint4(0, 0, 0, 0);
      amax = fmaxf(amax, absmax8_bf16(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) red[i & 1][warp] = amax;
    fence_proxy_async_smem();  // this thread's reads of the slot, before its async refill
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(err, DEVERR_TIMEOUT);
        // drain the copies still in flight (bounded) before the CTA exits
        for (int64_t j = i; j < nrows && j < i + R; ++j) mbar_wait(&full[j % R], uint32_t((j / R) & 1));
      }
      return;
    }
    if (tid == 0 && i + R < nrows) {
      mbar_arrive_expect_tx(&full[slot], row_bytes);
      bulk_load(ring + size_t(slot) * row_bytes, x + (row + R * G) * K8, row_bytes, &full[slot]);
    }
    float r = lane < nw ? red[i & 1][lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
    const float sc = __fdiv_rn(r, 127.0f);
    const float inv = __frcp_rn(sc);
    if (tid == 0) s[row] = sc;
    uint2* qr = q + row * K8;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int64_t idx = tid + 256 * j;
      if (idx < K8) {
        float f[8];
        unpack8(v[j], f);
        qr[idx] = quant8_i8(f, sc, inv);
      }
    }
  }
}

// One warp per row, for rows of up to 32 * VPL 16-byte vectors (K <= 4096 at
// VPL = 16): every load of the row is issued before its absmax is needed,
// the absmax is a warp shuffle reduction (no block barrier), and the CTA's
// WARPS warps keep as many rows in flight - at K = 4096, 12 rows (96 KB) per
// SM, enough to cover loaded HBM latency.
template <int VPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) quant_int8_warp_kernel(const uint4* __restrict__ x, int64_t M, int64_t K8,
                                                               uint2* __restrict__ q, float* __restrict__ s,
                                                               int trigger) {
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
  for (int64_t row = int64_t(blockIdx.x) * warps + (threadIdx.x >> 5); row < M; row += int64_t(gridDim.x) * warps) {
    const uint4* xr = x + row * K8;
    uint4 v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int64_t idx = lane + 32 * i;
      v[i] = idx < K8 ? ld_stream(xr + idx) : make_uint4(0, 0, 0, 0);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) amax = fmaxf(amax, absmax8_bf16(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float sc = __fdiv_rn(amax, 127.0f);
    const float inv = __frcp_rn(sc);
    if (lane == 0) s[row] = sc;
    uint2* qr = q + row * K8;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int64_t idx = lane + 32 * i;
      if (idx < K8) {
        float f[8];
        unpack8(v[i], f);
        qr[idx] = quant8_i8(f, sc, inv);
      }
    }
  }
}

// Small M: each row split along K over a cluster of CS CTAs (one 16-byte
// vector per thread), so M = 1..8 rows occupy CS * M SMs.  Each CTA reduces
// its slice, writes its partial absmax into every cluster member's shared
// memory (distributed shared memory), and after one cluster barrier each
// takes the max of the CS partials - the same value in every member - and
// quantizes its slice.  CTA rank 0 writes the scale.
template <int CS>
__global__ void __launch_bounds__(256) quant_int8_split_kernel(const uint4* __restrict__ x, int64_t M, int64_t K8,
                                                                uint2* __restrict__ q, float* __restrict__ s,
                                                                int trigger) {
  __shared__ float part[CS];
  __shared__ float red[8];
  // every member has started before anyone writes into its shared memory
  cluster_arrive_relaxed();
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / CS;
  const int64_t per = (K8 + CS - 1) / CS;  // vectors per member
  const int64_t idx = int64_t(rank) * per + threadIdx.x;
  const bool mine = threadIdx.x < per && idx < K8 && row < M;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (mine) v = ld_stream(x + row * K8 + idx);
  float f[8];
  unpack8(v, f);
  float amax = absmax8(f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  cluster_wait_acquire();
  if (threadIdx.x < CS) {
    float m = 0.0f;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    st_cluster_u32(mapa_shared(smem_u32(&part[rank]), uint32_t(threadIdx.x)), __float_as_uint(m));
  }
  cluster_sync_all();  // partials delivered (release / acquire across the cluster)
  float tot = 0.0f;
#pragma unroll
  for (int c = 0; c < CS; ++c) tot = fmaxf(tot, part[c]);
  const float sc = __fdiv_rn(tot, 127.0f);
  const float inv = __frcp_rn(sc);
  if (row < M) {
    if (rank == 0 && threadIdx.x == 0) s[row] = sc;
    if (mine) q[row * K8 + idx] = quant8_i8(f, sc, inv);
  }
}

// ---------------------------------------------------------------- a7: SwiGLU + INT8

// h = bf16_RN(fp32(s * u)) with s = fp32_RN(silu(g)), silu(g) = g / (1 + exp(-g))
// rounded once to fp32 (the exact value's rounding); then the per-token
// quant of h.  One CTA per row; VPT vectors of 8 outputs cached.
//
// Fast path: s is estimated in fp32 with expf.  For |g| <= 64 that estimate
// is within 5 units in the last place of the correctly rounded s (expf's
// documented 2-ulp bound plus at most three fp32 roundings, all on normal
// numbers), so the correctly rounded s lies in the bracket of +-16 ulp steps
// around it (twice the bound, for a bracket that crosses a power of two).
// h is a monotone function of s for a fixed u (two monotone roundings of a
// product), so when both ends of the bracket give the same h, that h is
// exact.  Otherwise (h within a few fp32 ulps of a bf16 rounding boundary,
// about 5e-4 of elements, or |g| > 64) s is recomputed as the fp64 quotient
// g / (1 + exp(-g)) rounded once to fp32.  For all but 32 bf16 values of g
// (all with |g| < 6e-5) silu(g) lies more than 2^-45 (relative) from every
// fp32 rounding midpoint, far beyond the fp64 quotient's error, so this is
// the correctly rounded s; for those 32 the fp64 steps are the same IEEE
// operations on an argument whose exp any fp64 library rounds correctly.
// Tests check every bf16 g.
__device__ __forceinline__ uint16_t swiglu_h_bits(float g, float u) {
  // silu(g) = g / (1 + e^-g); for g < 0 the same value as g e^g / (1 + e^g),
  // which does not overflow for large |g|
  float sg;
  if (g >= 0.0f) {
    sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  } else {
    const float e = expf(g);
    sg = __fdiv_rn(__fmul_rn(g, e), __fadd_rn(1.0f, e));
  }
  if (fabsf(g) <= 64.0f) {
    const uint32_t b = __float_as_uint(sg);
    const uint32_t sign = b & 0x80000000u, mag = b & 0x7FFFFFFFu;
    const float s_lo = __uint_as_float(sign | (mag > 16u ? mag - 16u : 0u));
    const float s_hi = __uint_as_float(sign | (mag + 16u));
    const uint16_t h_lo = f32_to_bf16_bits(__fmul_rn(s_lo, u));
    const uint16_t h_hi = f32_to_bf16_bits(__fmul_rn(s_hi, u));
    if (h_lo == h_hi) return h_lo;
  }
  const double gd = double(g);
  const float s = __double2float_rn(__ddiv_rn(gd, __dadd_rn(1.0, exp(-gd))));
  return f32_to_bf16_bits(__fmul_rn(s, u));
}

__device__ __forceinline__ void swiglu8(const uint4& gv, const uint4& uv, float h[8], uint4* hbits) {
  float g[8], u[8];
  unpack8(gv, g);
  unpack8(uv, u);
  uint32_t hb[4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint16_t b = swiglu_h_bits(g[i], u[i]);
    h[i] = __uint_as_float(uint32_t(b) << 16);
    if (i & 1)
      hb[i >> 1] |= uint32_t(b) << 16;
    else
      hb[i >> 1] = b;
  }
  *hbits = make_uint4(hb[0], hb[1], hb[2], hb[3]);
}

template <int VPT>
__global__ void __launch_bounds__(256) swiglu_quant_int8_kernel(const uint4* __restrict__ gu, int64_t rows,
                                                                 int64_t I8, uint2* __restrict__ hq,
                                                                 float* __restrict__ sh, uint4* __restrict__ hout) {
  __shared__ float red[32];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint4* gr = gu + row * 2 * I8;
    const uint4* ur = gr + I8;
    float h[VPT][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      if (idx < I8) {
        uint4 hb;
        swiglu8(ld_stream(gr + idx), ld_stream(ur + idx), h[i], &hb);
        if (hout) hout[row * I8 + idx] = hb;
        amax = fmaxf(amax, absmax8(h[i]));
      }
    }
    for (int64_t idx = tid + int64_t(VPT) * nt; idx < I8; idx += nt) {
      float t[8];
      uint4 hb;
      swiglu8(gr[idx], ur[idx], t, &hb);
      if (hout) hout[row * I8 + idx] = hb;
      amax = fmaxf(amax, absmax8(t));
    }
    amax = block_max(amax, red);
    const float sc = __fdiv_rn(amax, 127.0f);
    const float inv = __frcp_rn(sc);
    if (tid == 0) sh[row] = sc;
    uint2* qr = hq + row * I8;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * nt;
      if (idx < I8) qr[idx] = quant8_i8(h[i], sc, inv);
    }
    for (int64_t idx = tid + int64_t(VPT) * nt; idx < I8; idx += nt) {
      float t[8];
      uint4 hb;
      swiglu8(gr[idx], ur[idx], t, &hb);
      qr[idx] = quant8_i8(t, sc, inv);
    }
  }
}

// ---------------------------------------------------------------- a5: gather

// Row i of the expert-ordered copy is source token perm[i] / topk.
__global__ void __launch_bounds__(256) gather_rows_i8_kernel(const uint4* __restrict__ xq, const float* __restrict__ sx,
                                                              const int32_t* __restrict__ perm, int64_t R,
                                                              int64_t topk, int64_t K16, int64_t T,
                                                              uint4* __restrict__ xg, float* __restrict__ sg) {
  pdl_wait();
  pdl_launch_dependents();
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t row = int64_t(blockIdx.x) * warps + warp; row < R; row += int64_t(gridDim.x) * warps) {
    int64_t src = perm[row] / topk;
    if (src < 0 || src >= T) src = 0;  // perm comes from moe_sort; stay in bounds regardless
    if (lane == 0) sg[row] = sx[src];
    for (int64_t c = lane; c < K16; c += 32) xg[row * K16 + c] = xq[src * K16 + c];
  }
}

// ---------------------------------------------------------------- a3: FP8 group quant

// e = clamp(ceil(log2(amax / 448)), -127, 127) from the bits of amax:
// with amax = 1.f * 2^E, amax <= 448 * 2^k  <=>  1.f <= 1.75 * 2^(k + 8 - E),
// so k = E - 8 when the fraction 1.f <= 1.75 (mantissa bits <= 0x600000) and
// E - 7 otherwise.  Zero and subnormal amax fall below the clamp (-127).
__device__ __forceinline__ int ue8m0_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int E = int((b >> 23) & 0xFFu);
  if (E == 0) return -127;
  const int e = (E - 127) - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return max(-127, min(127, e));
}

// 2^e as fp32 for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_int(int e) {
  const int be = e + 127;
  return be >= 1 ? __uint_as_float(uint32_t(be) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// One warp per (t, g, pack p) unit: lanes 8i..8i+7 cover hidden group
// j = 4p + i (16 elements each, two 16-byte loads), an 8-lane shuffle gives
// the group absmax, and lane 0 assembles the four exponent bytes into one
// int32 word.  Groups past NG contribute byte 0 (zeroed tail of the last
// pack); token-padding units t >= T write a zero word and touch no payload.
// PACKED = false writes fp32 scales [T, G, NG] instead (the A/B control).
template <bool PACKED>
__global__ void __launch_bounds__(256) quant_fp8_group_kernel(const uint4* __restrict__ x, int T, int G, int NG,
                                                               int P, int Ta, uint4* __restrict__ xq,
                                                               int32_t* __restrict__ s_packed,
                                                               float* __restrict__ s_f32) {
  pdl_wait();
  pdl_launch_dependents();
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane >> 3, l8 = lane & 7;
  const int64_t D16 = int64_t(NG) * 16;  // 16-byte vectors of bf16 per (t, g) row (8 elem each)
  const int64_t units = PACKED ? int64_t(G) * P * Ta : int64_t(G) * P * T;
  // 32-bit unit decode when the units fit (GB300, T=4096, G=8, D=4096: 80.4
  // -> 78.8 us against 64-bit div/mod per unit)
  const bool narrow = units <= int64_t(UINT32_MAX);
  for (int64_t u = int64_t(blockIdx.x) * warps + warp; u < units; u += int64_t(gridDim.x) * warps) {
    // unit order follows the scale words: ((g * P + p) * Ta + t)
    const int tdim = PACKED ? Ta : T;
    int t, p, g;
    if (narrow) {
      const uint32_t uu = uint32_t(u), gp = uu / uint32_t(tdim);
      t = int(uu - gp * uint32_t(tdim));
      g = int(gp / uint32_t(P));
      p = int(gp - uint32_t(g) * uint32_t(P));
    } else {
      const int64_t gp = u / tdim;
      t = int(u - gp * tdim);
      p = int(gp % P);
      g = int(gp / P);
    }
    const int j = 4 * p + sub;
    // every lane joins the shuffles; lanes past the last group or in token
    // padding carry zeros and store nothing
    const bool active = (t < T) && (j < NG);
    const int64_t vbase = (int64_t(t) * G + g) * D16 + int64_t(j) * 16 + l8 * 2;
    float f[16];
    if (active) {
      const uint4 v0 = ld_stream(x + vbase), v1 = ld_stream(x + vbase + 1);
      unpack8(v0, f);
      unpack8(v1, f + 8);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int e = ue8m0_exp(amax);
    uint32_t byte = 0;
    if (active) {
      const float sc = exp2_int(-e);
      uint4 o;
      o.x = e4m3x4(f[0] * sc, f[1] * sc, f[2] * sc, f[3] * sc);
      o.y = e4m3x4(f[4] * sc, f[5] * sc, f[6] * sc, f[7] * sc);
      o.z = e4m3x4(f[8] * sc, f[9] * sc, f[10] * sc, f[11] * sc);
      o.w = e4m3x4(f[12] * sc, f[13] * sc, f[14] * sc, f[15] * sc);
      xq[vbase / 2] = o;  // 16 E4M3 codes = one uint4 per lane
      byte = uint32_t(e + 127);
      if (!PACKED && l8 == 0) s_f32[(int64_t(t) * G + g) * NG + j] = exp2_int(e);
    }
    if (PACKED) {
      const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, 8);
      const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, 16);
      const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, 24);
      if (lane == 0) s_packed[u] = int32_t(byte | (b1 << 8) | (b2 << 16) | (b3 << 24));
    }
  }
}

// ---------------------------------------------------------------- RMSNorm + quant producer
//
// "Reshaping LLM inference dataflow: DeepSeek V4 950" section 2.3, first
// fusion: normalise in registers and write only the quantized activation.
// One CTA (256 threads) per row, each thread holding VPT 16-byte vectors.
//   ss = sum x^2, rounded once to fp64 from an integer sum: a bf16 value is
//        an 8-bit integer mantissa times a power of two, so every x^2 is a
//        16-bit integer shifted by twice its exponent; aligned to the row's
//        largest exponent with a 96-bit window the terms add exactly in a
//        128-bit integer, and bits below the window only set a sticky bit
//        (their total is below 2^-82 of the sum; the sticky bit keeps the
//        fp64 rounding of ties exact);
//   r  = fp32(1 / sqrt(ss / K + eps)) in IEEE fp64 steps (r = 0 if the
//        argument is 0);
//   y  = fp32(fp32(x * r) * gamma), then the INT8 per-token rule or the FP8
//        per-128-group rule with packed UE8M0 scales (one outer group).
typedef unsigned __int128 u128;

// x^2 of a bf16-valued float in units of 2^(2*(emax - 134) - 96), where emax
// is the row's largest biased exponent (subnormals count as exponent 1).
// Bits that fall below the window are dropped and reported in `sticky`; the
// caller ORs them into the lowest unit of the sum, which lies far below the
// fp64 rounding position, so a rounding tie is broken as the exact sum would.
__device__ __forceinline__ u128 sq_units(float v, int emax, uint32_t& sticky) {
  const uint32_t b = __float_as_uint(v);
  const int ex = int((b >> 23) & 0xFFu);
  const uint32_t m = ((b >> 16) & 0x7Fu) | (ex ? 0x80u : 0u);  // the 8-bit integer mantissa
  const int d = 2 * (emax - (ex ? ex : 1));
  const uint64_t m2 = uint64_t(m) * m;  // < 2^16
  if (d <= 96) return u128(m2) << (96 - d);
  const int sh = d - 96;
  if (sh >= 16) {
    sticky |= (m2 != 0);
    return 0;
  }
  sticky |= ((m2 & ((1ull << sh) - 1)) != 0);
  return u128(m2 >> sh);
}

// Correctly rounded fp64 value of S * 2^k (S > 0): the top 64 bits of S with
// a sticky bit for anything below, converted with one rounding, then an
// exact power-of-two scaling.
__device__ __forceinline__ double u128_to_f64_scaled(u128 S, int k) {
  const uint64_t hi = uint64_t(S >> 64), lo = uint64_t(S);
  uint64_t top;
  int shift;
  if (hi) {
    const int lz = __clzll(hi);
    shift = 64 - lz;  // bits dropped below the top 64
    top = (hi << lz) | (lz ? (lo >> (64 - lz)) : 0ull);
    const uint64_t rest = lz ? (lo << lz) : lo;
    if (rest) top |= 1ull;
  } else {
    top = lo;
    shift = 0;
  }
  const double t = __ull2double_rn(top);
  const int e = k + shift;  // within fp64's normal range for any bf16 row
  return __dmul_rn(t, __longlong_as_double(int64_t(e + 1023) << 52));
}

template <int VPT, bool FP8>
__global__ void __launch_bounds__(256) rmsnorm_quant_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                                                             float eps, int64_t rows, int64_t T, int64_t K8,
                                                             uint2* __restrict__ q, float* __restrict__ sx,
                                                             int32_t* __restrict__ s_packed, int P, int Ta) {
  __shared__ uint64_t red_hi[8], red_lo[8];
  __shared__ uint32_t red_sticky[8];
  __shared__ float red[32];
  __shared__ float s_r;
  __shared__ uint8_t s_bytes[(FP8 ? VPT * 256 / 16 : 1) + 4];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    if (FP8 && row >= T) {  // token padding of the packed scales: zero words
      for (int p = tid; p < P; p += 256) s_packed[int64_t(p) * Ta + row] = 0;
      continue;
    }
    const uint4* xr = x + row * K8;
    float f[VPT][8];
    float xmax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * 256;
      if (idx < K8) {
        unpack8(ld_stream(xr + idx), f[i]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[i][k] = 0.0f;
      }
      xmax = fmaxf(xmax, absmax8(f[i]));
    }
    xmax = block_max(xmax, red);
    const int emax_raw = int((__float_as_uint(xmax) >> 23) & 0xFFu);
    const int emax = emax_raw ? emax_raw : 1;
    u128 acc = 0;
    uint32_t sticky = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc += sq_units(f[i][k], emax, sticky);
    sticky = __any_sync(0xFFFFFFFFu, sticky != 0);
    uint64_t ahi = uint64_t(acc >> 64), alo = uint64_t(acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const u128 other = (u128(__shfl_xor_sync(0xFFFFFFFFu, ahi, o)) << 64) | __shfl_xor_sync(0xFFFFFFFFu, alo, o);
      const u128 sum = ((u128(ahi) << 64) | alo) + other;
      ahi = uint64_t(sum >> 64);
      alo = uint64_t(sum);
    }
    if (lane == 0) {
      red_hi[warp] = ahi;
      red_lo[warp] = alo;
      red_sticky[warp] = sticky;
    }
    __syncthreads();
    if (tid == 0) {
      u128 S = 0;
      uint32_t st_any = 0;
      for (int w = 0; w < 8; ++w) {
        S += (u128(red_hi[w]) << 64) | red_lo[w];
        st_any |= red_sticky[w];
      }
      if (st_any) S |= 1u;
      const double ss = S == 0 ? 0.0 : u128_to_f64_scaled(S, 2 * (emax - 134) - 96);
      const double u = __dadd_rn(__ddiv_rn(ss, double(K8 * 8)), double(eps));
      s_r = (u == 0.0) ? 0.0f : __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn(u)));
    }
    __syncthreads();
    const float r = s_r;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t idx = tid + int64_t(i) * 256;
      if (idx < K8) {
        float g[8];
        unpack8(__ldg(gamma + idx), g);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[i][k] = __fmul_rn(__fmul_rn(f[i][k], r), g[k]);
      }
      if (!FP8) amax = fmaxf(amax, absmax8(f[i]));
    }
    uint2* qr = q + row * K8;
    if (!FP8) {
      amax = block_max(amax, red);
      const float sc = __fdiv_rn(amax, 127.0f);
      const float inv = __frcp_rn(sc);
      if (tid == 0) sx[row] = sc;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int64_t idx = tid + int64_t(i) * 256;
        if (idx < K8) qr[idx] = quant8_i8(f[i], sc, inv);
      }
    } else {
      // a 128-element group is 16 consecutive vectors: 16 consecutive threads
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int64_t idx = tid + int64_t(i) * 256;
        float ga = absmax8(f[i]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ga = fmaxf(ga, __shfl_xor_sync(0xFFFFFFFFu, ga, o));
        if (idx < K8) {
          const int e = ue8m0_exp(ga);
          const float sc = exp2_int(-e);
          uint2 o;
          o.x = e4m3x4(f[i][0] * sc, f[i][1] * sc, f[i][2] * sc, f[i][3] * sc);
          o.y = e4m3x4(f[i][4] * sc, f[i][5] * sc, f[i][6] * sc, f[i][7] * sc);
          qr[idx] = o;
          if ((idx & 15) == 0) s_bytes[idx >> 4] = uint8_t(e + 127);
        }
      }
      __syncthreads();
      const int NG = int(K8 >> 4);
      for (int p = tid; p < P; p += 256) {
        uint32_t w = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (4 * p + b < NG) w |= uint32_t(s_bytes[4 * p + b]) << (8 * b);
        s_packed[int64_t(p) * Ta + row] = int32_t(w);
      }
    }
    __syncthreads();  // shared scratch is reused by the next row
  }
}

// ---------------------------------------------------------------- 32-element block-scaled FP8
//
// "Reshaping LLM inference dataflow: DeepSeek V4 950" section 2.1: 32
// elements share one 8-bit (UE8M0) scale with E4M3 payloads.  One thread per
// 8-element vector, 4 consecutive lanes per 32-element block (a shuffle
// gives the block absmax).  The scale bytes are written in the blocked layout
// the linear's tensor-core scale copy reads: for every 128 rows x 128 K one
// 512-byte chunk, row r's byte for K block b at
// (r % 32) * 16 + ((r % 128) / 32) * 4 + b % 4.
template <int U>
__global__ void __launch_bounds__(256) quant_mxfp8_kernel(const uint4* __restrict__ x, int64_t R, int64_t K8,
                                                          uint2* __restrict__ q, uint8_t* __restrict__ sf) {
  // no early trigger: the output is the weight operand of a linear as often
  // as its activations, and a dependent may read its weights before its own
  // wait
  pdl_wait();
  const int64_t total = R * K8, KB = K8 / 16;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t span = (total + 31) / 32 * 32;  // whole warps stay in the loop together
  // U vectors a thread per pass, their loads issued first: with many rows one
  // 16-byte load in flight per thread leaves HBM short of requests
  for (int64_t v0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v0 - threadIdx.x % 32 < span; v0 += U * stride) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      raw[u] = v < total ? ld_stream(x + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * stride;
      const bool ok = v < total;
      float f[8];
      unpack8(raw[u], f);
      float amax = absmax8(f);
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
      if (ok) {
        const int e = ue8m0_exp(amax);
        const float sc = exp2_int(-e);
        uint2 o;
        o.x = e4m3x4(f[0] * sc, f[1] * sc, f[2] * sc, f[3] * sc);
        o.y = e4m3x4(f[4] * sc, f[5] * sc, f[6] * sc, f[7] * sc);
        q[v] = o;
        if ((v & 3) == 0) {
          const int64_t r = v / K8, b = (v - r * K8) >> 2;
          sf[((r >> 7) * KB + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)] = uint8_t(e + 127);
        }
      }
    }
  }
  // rows R .. 128*ceil(R/128)-1 of the last chunk row hold zero bytes
  const int64_t pad_rows = (R + 127) / 128 * 128 - R;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < pad_rows * KB * 4; i += stride) {
    const int64_t r = R + i / (KB * 4), b = i % (KB * 4);
    sf[((r >> 7) * KB + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)] = 0;
  }
}

// fp32 power-of-two scales [T, G, NG] -> packed int32 [G, P, Ta]; one thread per word.
__global__ void __launch_bounds__(256) pack_scales_kernel(const float* __restrict__ s, int T, int G, int NG, int P,
                                                           int Ta, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t words = int64_t(G) * P * Ta;
  for (int64_t w = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; w < words; w += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(w % Ta);
    const int64_t gp = w / Ta;
    const int p = int(gp % P), g = int(gp / P);
    uint32_t word = 0;
    if (t < T) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int j = 4 * p + b;
        if (j < NG) {
          const uint32_t bits = __float_as_uint(s[(int64_t(t) * G + g) * NG + j]) & 0x7FFFFFFFu;
          const int E = int(bits >> 23);
          // a power of two: normal -> E - 127; subnormal 2^k -> k = log2(mantissa) - 149
          const int e = E ? (E - 127) : ((31 - __clz(bits)) - 149);
          word |= uint32_t(max(-127, min(127, e)) + 127) << (8 * b);
        }
      }
    }
    out[w] = int32_t(word);
  }
}

// ---------------------------------------------------------------- fp8 weight prep

// One CTA per 128 x 128 block (rows n, columns d of w[G, N, D]).
__global__ void __launch_bounds__(256) quantize_weight_fp8_kernel(const float4* __restrict__ w, int G, int N, int D,
                                                                   uint32_t* __restrict__ wq, float* __restrict__ sw) {
  __shared__ float red[32];
  const int NB = N / 128, KB = D / 128;
  const int b = blockIdx.x;
  const int kb = b % KB, nb = (b / KB) % NB, g = b / (KB * NB);
  const int tid = threadIdx.x;
  const int64_t D4 = D / 4;
  float4 v[16];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int f4 = tid + i * 256;           // 0..4095 float4 of the block
    const int r = f4 >> 5, c4 = f4 & 31;    // 32 float4 per 128-wide row
    v[i] = w[(int64_t(g) * N + nb * 128 + r) * D4 + kb * 32 + c4];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 448.0f);
  if (tid == 0) sw[(int64_t(g) * KB + kb) * NB + nb] = s;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int f4 = tid + i * 256;
    const int r = f4 >> 5, c4 = f4 & 31;
    float a = 0.f, bb = 0.f, c = 0.f, d = 0.f;
    if (s != 0.0f) {
      a = __fdiv_rn(v[i].x, s);
      bb = __fdiv_rn(v[i].y, s);
      c = __fdiv_rn(v[i].z, s);
      d = __fdiv_rn(v[i].w, s);
    }
    wq[(int64_t(g) * N + nb * 128 + r) * D4 + kb * 32 + c4] = e4m3x4(a, bb, c, d);
  }
}

static int grid_for(int64_t work, int per_cta, int sms, int ctas_per_sm) {
  int64_t need = (work + per_cta - 1) / per_cta;
  int64_t cap = int64_t(sms) * ctas_per_sm;
  return int(need < cap ? (need > 0 ? need : 1) : cap);
}

// CTAs of `kernel` an SM holds at once (registers, threads, shared memory),
// at most `cap`.  A grid-stride kernel sized to this runs in one wave: a grid
// of more CTAs than the SMs hold leaves a partial second wave, and the next
// kernel's early-launched CTAs, parked at their dependency wait, then take
// the slots that wave needs.  Cached per (kernel, block size).
static int resident_ctas(const void* kernel, int threads, int cap) {
  struct Entry {
    const void* k;
    int threads, n;
  };
  static Entry tab[64];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int n = 0;
  for (int i = 0; i < used && !n; ++i)
    if (tab[i].k == kernel && tab[i].threads == threads) n = tab[i].n;
  if (!n) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    if (used < 64) tab[used++] = {kernel, threads, n};
  }
  return n < cap ? n : cap;
}

// the grid of a grid-stride kernel over `work` units (`per_cta` a CTA at a time), one wave
template <typename Kern>
static int wave_grid(Kern kernel, int threads, int64_t work, int per_cta, int sms, int cap) {
  return grid_for(work, per_cta, sms, resident_ctas(reinterpret_cast<const void*>(kernel), threads, cap));
}

}  // namespace fq

using namespace fq;

// ================================================================ entry points

// Kernel choice for the per-token INT8 quant (FQ_QUANT_KERNEL = wide | row |
// ring | warp | split overrides it; tests and studies).  Measured on GB300,
// each call in a CUDA graph (us per call at M = 1..64, K = 4096 / K = 1024;
// M = 16384, K = 4096):
//  * few rows (M <= SM count): one CTA per row with up to 1024 threads, one
//    16-byte vector a thread for K <= 8192 ("wide"): 1.96-2.15 / 1.79-2.06.
//    A decode-sized row is one round trip to memory; what remains on the
//    critical path is the per-thread quant arithmetic and the block barrier.
//  * many rows: CTAs of 256 threads (128 for 2048 < K <= 4096), grid-stride
//    over rows, the next row's loads in flight while the current one is
//    reduced and stored ("row"): 44 us at M = 16384 (0.67 of HBM; 60 us
//    before the packed-pair absmax, the eight-at-a-time code path and the
//    128-thread rows - the kernel is issue-bound, ~21 instructions an element
//    at 256 threads, a third of them per-row reduction and scale).
//  * built, tested, taken only when forced: 256-thread rows without the
//    prefetch (2.35-2.8 / 1.82-2.2; 66.5 us), rows staged through a
//    shared-memory ring by bulk copies 8-16 rows ahead ("ring", 70 us), one
//    warp per row ("warp": a lane quantizes 128 values one after the other,
//    7.2 us at M = 1) and the row split along K over a cluster with a
//    distributed-shared-memory absmax exchange ("split", M <= 8: 2.1-2.45 /
//    2.15-2.4 - the cluster barriers cost what the split saves).
enum QuantKernel { QK_AUTO = 0, QK_WIDE = 1, QK_ROW = 2, QK_WARP = 3, QK_SPLIT = 4, QK_RING = 5 };
static int forced_quant_kernel() {
  const char* v = std::getenv("FQ_QUANT_KERNEL");
  if (!v) return QK_AUTO;
  if (!std::strcmp(v, "wide")) return QK_WIDE;
  if (!std::strcmp(v, "row")) return QK_ROW;
  if (!std::strcmp(v, "warp")) return QK_WARP;
  if (!std::strcmp(v, "split")) return QK_SPLIT;
  if (!std::strcmp(v, "ring")) return QK_RING;
  return QK_AUTO;
}

fq_status fq::quant_int8_launch(const uint16_t* x, int64_t M, int64_t K, int8_t* xq, float* sx, fq_stream_t stream,
                            bool trigger) {
  if (M < 0 || K < 0 || K % 16 || K > (int64_t(1) << 30) || M > (int64_t(1) << 40)) return FQ_ERR_SHAPE;
  if (M == 0) return FQ_OK;
  if (!x || !xq || !sx) return FQ_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(sx)) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t K8 = K / 8;
  const bool pdl = pdl_enabled();
  cudaError_t e;
  auto xp = reinterpret_cast<const uint4*>(x);
  auto qp = reinterpret_cast<uint2*>(xq);
  const int tr = trigger ? 1 : 0;
  int force = forced_quant_kernel();
  if (force == QK_SPLIT && !(M <= 8 && K8 > 0 && K8 <= 2048)) force = QK_AUTO;
  if (force == QK_WARP && K8 > 512) force = QK_AUTO;
  if (force == QK_RING && !(K8 > 0 && K8 <= 1024)) force = QK_AUTO;
  if (force == QK_WIDE && K8 > 4096) force = QK_AUTO;
  if (force == QK_ROW && K8 > 1024) force = QK_AUTO;
  if (force == QK_AUTO) force = M <= d.sm_count ? (K8 <= 4096 ? QK_WIDE : QK_AUTO) : (K8 <= 1024 ? QK_ROW : QK_AUTO);
  if (force == QK_SPLIT) {
    // 8 CTAs per row when each gets at least 64 vectors, else 4 or 2
    const int cs = K8 >= 512 ? 8 : (K8 >= 256 ? 4 : 2);
    const int64_t per = (K8 + cs - 1) / cs;
    const int threads = per > 128 ? 256 : (per > 64 ? 128 : (per > 32 ? 64 : 32));
    const int grid = int(M) * cs;
    e = cs == 8 ? launch_cluster(quant_int8_split_kernel<8>, grid, threads, 0, s, pdl, 8u, xp, M, K8, qp, sx, tr)
        : cs == 4 ? launch_cluster(quant_int8_split_kernel<4>, grid, threads, 0, s, pdl, 4u, xp, M, K8, qp, sx, tr)
                  : launch_cluster(quant_int8_split_kernel<2>, grid, threads, 0, s, pdl, 2u, xp, M, K8, qp, sx, tr);
    return cuda_status(e);
  }
  if (force == QK_WARP) {
    const int vpl = int((K8 + 31) / 32);
    const int warps = vpl > 8 ? 12 : 16;  // registers: 16 vectors a lane hold 64 of them
    const int64_t ctas = (M + warps - 1) / warps;
    const int grid = int(ctas < int64_t(d.sm_count) * 2 ? ctas : int64_t(d.sm_count) * 2);
    if (vpl <= 1)
      e = launch(quant_int8_warp_kernel<1, 16>, grid, 32 * warps, 0, s, pdl, xp, M, K8, qp, sx, tr);
    else if (vpl <= 2)
      e = launch(quant_int8_warp_kernel<2, 16>, grid, 32 * warps, 0, s, pdl, xp, M, K8, qp, sx, tr);
    else if (vpl <= 4)
      e = launch(quant_int8_warp_kernel<4, 16>, grid, 32 * warps, 0, s, pdl, xp, M, K8, qp, sx, tr);
    else if (vpl <= 8)
      e = launch(quant_int8_warp_kernel<8, 16>, grid, 32 * warps, 0, s, pdl, xp, M, K8, qp, sx, tr);
    else
      e = launch(quant_int8_warp_kernel<16, 12>, grid, 32 * warps, 0, s, pdl, xp, M, K8, qp, sx, tr);
    return cuda_status(e);
  }
  if (force == QK_RING) {
    const size_t row_bytes = size_t(K8) * 16;
    int R = int(65536 / row_bytes);
    R = R < 2 ? 2 : (R > kRingMax ? kRingMax : R);
    const size_t smem = size_t(R) * row_bytes;
    const int grid = grid_for(M, 1, d.sm_count, 3);
    const int vpt = int((K8 + 255) / 256);
    auto k = vpt <= 1 ? quant_int8_ring_kernel<1> : (vpt <= 2 ? quant_int8_ring_kernel<2> : quant_int8_ring_kernel<4>);
    static uint64_t attr_done[3] = {0, 0, 0};
    const int ki = vpt <= 1 ? 0 : (vpt <= 2 ? 1 : 2);
    if (!(attr_done[ki] & (1ull << (d.id & 63)))) {
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536)) != cudaSuccess)
        return cuda_status(e);
      attr_done[ki] |= 1ull << (d.id & 63);
    }
    e = launch(k, grid, 256, smem, s, pdl, xp, M, K8, qp, sx, tr, R, d.err_word);
    return cuda_status(e);
  }
  if (force == QK_WIDE || force == QK_ROW) {
    // WIDE: up to 1024 threads, one vector each while K <= 8192; ROW: 256 threads
    const int64_t t32 = (K8 + 31) / 32 * 32;
    const int threads = force == QK_ROW ? (K8 >= 256 ? 256 : int(t32)) : int(t32 < 1024 ? t32 : 1024);
    const int64_t vpt = (K8 + threads - 1) / threads;
    if (force == QK_ROW) {
      if (K8 > 256 && K8 <= 512) {
        // 128 threads, four vectors each: the per-row reduction and scale
        // spread over twice the elements (the kernel is issue-bound: 50 -> 44 us
        // at M=16384, K=4096 on GB300)
        const int grid = grid_for(M, 1, d.sm_count, 8);
        e = launch(quant_int8_stream_kernel<4, 128, 8>, grid, 128, 0, s, pdl, xp, M, K8, qp, sx, tr);
        return cuda_status(e);
      }
      const int grid = grid_for(M, 1, d.sm_count, 6 * 256 / threads);
      if (vpt <= 1)
        e = launch(quant_int8_stream_kernel<1, 256, 6>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
      else if (vpt <= 2)
        e = launch(quant_int8_stream_kernel<2, 256, 6>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
      else
        e = launch(quant_int8_stream_kernel<4, 256, 6>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
    } else {
      const int grid = grid_for(M, 1, d.sm_count, 2048 / threads);
      if (vpt <= 1)
        e = launch(quant_int8_stream_kernel<1, 1024, 1>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
      else if (vpt <= 2)
        e = launch(quant_int8_stream_kernel<2, 1024, 1>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
      else
        e = launch(quant_int8_stream_kernel<4, 1024, 1>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
    }
    return cuda_status(e);
  }
  // long rows (K > 8192 with many rows, K > 32768 with few): one CTA per row
  // re-reading the part of the row its registers do not hold
  const int threads = 256;
  const int grid = grid_for(M, 1, d.sm_count, 2048 / threads);
  e = launch(dynamic_quant_int8_kernel<8>, grid, threads, 0, s, pdl, xp, M, K8, qp, sx, tr);
  return cuda_status(e);
}

extern "C" __attribute__((visibility("default"))) fq_status dynamic_quant_int8(const uint16_t* x, int64_t M, int64_t K, int8_t* xq, float* sx,
                                        fq_stream_t stream) {
  return quant_int8_launch(x, M, K, xq, sx, stream, false);
}

extern "C" __attribute__((visibility("default"))) fq_status swiglu_quant_int8(const uint16_t* gu, int64_t rows, int64_t I, int8_t* hq, float* sh,
                                       uint16_t* h_out, fq_stream_t stream) {
  if (rows < 0 || I < 0 || I % 16 || I > (int64_t(1) << 28)) return FQ_ERR_SHAPE;
  if (rows == 0 || I == 0) return FQ_OK;
  if (!gu || !hq || !sh) return FQ_ERR_NULL;
  if (!aligned16(gu) || !aligned16(hq) || !aligned16(sh) || (h_out && !aligned16(h_out))) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t I8 = I / 8;
  const int threads = I8 >= 256 ? 256 : (I8 >= 128 ? 128 : (I8 >= 64 ? 64 : 32));
  const int64_t vpt = (I8 + threads - 1) / threads;
  const bool pdl = pdl_enabled();
  auto gp = reinterpret_cast<const uint4*>(gu);
  auto qp = reinterpret_cast<uint2*>(hq);
  auto hp = reinterpret_cast<uint4*>(h_out);
  // More CTAs than the SMs hold at once: one row per CTA at a time, so the
  // extra rows in flight pay (a one-wave grid measured 20.3 -> 21.6 us at
  // 2048 rows, I = 2048, on GB300).
  const int grid = grid_for(rows, 1, d.sm_count, 2048 / threads);
  cudaError_t e;
  if (vpt <= 1)
    e = launch(swiglu_quant_int8_kernel<1>, grid, threads, 0, s, pdl, gp, rows, I8, qp, sh, hp);
  else if (vpt <= 2)
    e = launch(swiglu_quant_int8_kernel<2>, grid, threads, 0, s, pdl, gp, rows, I8, qp, sh, hp);
  else
    e = launch(swiglu_quant_int8_kernel<4>, grid, threads, 0, s, pdl, gp, rows, I8, qp, sh, hp);
  return cuda_status(e);
}

extern "C" __attribute__((visibility("default"))) fq_status moe_gather_rows_i8(const int8_t* xq, const float* sx, const int32_t* perm, int64_t T,
                                        int64_t topk, int64_t K, int8_t* xq_g, float* sx_g, fq_stream_t stream) {
  if (T < 0 || topk <= 0 || K < 0 || K % 16 || T * topk > (int64_t(1) << 31)) return FQ_ERR_SHAPE;
  const int64_t R = T * topk;
  if (R == 0) return FQ_OK;
  if (!xq || !sx || !perm || !xq_g || !sx_g) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(xq_g) || !aligned16(perm) || !aligned16(sx) || !aligned16(sx_g))
    return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int grid = grid_for(R, 8, d.sm_count, 8);
  return cuda_status(launch(gather_rows_i8_kernel, grid, 256, 0, reinterpret_cast<cudaStream_t>(stream),
                            pdl_enabled(), reinterpret_cast<const uint4*>(xq), sx, perm, R, topk, K / 16, T,
                            reinterpret_cast<uint4*>(xq_g), sx_g));
}

static fq_status fp8_group_common(const uint16_t* x, int64_t T, int64_t G, int64_t D, uint8_t* xq, int32_t* sp,
                                  float* sf, fq_stream_t stream, bool packed) {
  if (T < 0 || G < 0 || D < 0 || D % 128 || T > (int64_t(1) << 30) || G > (int64_t(1) << 20) ||
      D > (int64_t(1) << 24))
    return FQ_ERR_SHAPE;
  const int64_t NG = D / 128, P = (NG + 3) / 4, Ta = (T + 3) / 4 * 4;
  if (G == 0 || D == 0 || T == 0) return FQ_OK;  // T == 0: the [G, P, 0] storage is empty
  if (!x || !xq || (packed ? !sp : !sf)) return FQ_ERR_NULL;
  if (!aligned16(x) || !aligned16(xq) || (sp && !aligned16(sp)) || (sf && !aligned16(sf))) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t units = G * P * (sp ? Ta : T);
  if (units == 0) return FQ_OK;
  // one wave (GB300, T=4096, G=8, D=4096: 39 registers hold 6 CTAs of 256 per SM;
  // 8 per SM measured 79.2 against 69.5 us)
  const int grid = sp ? wave_grid(quant_fp8_group_kernel<true>, 256, units, 8, d.sm_count, 8)
                      : wave_grid(quant_fp8_group_kernel<false>, 256, units, 8, d.sm_count, 8);
  cudaError_t e;
  if (sp)
    e = launch(quant_fp8_group_kernel<true>, grid, 256, 0, s, pdl_enabled(), reinterpret_cast<const uint4*>(x),
               int(T), int(G), int(NG), int(P), int(Ta), reinterpret_cast<uint4*>(xq), sp, (float*)nullptr);
  else
    e = launch(quant_fp8_group_kernel<false>, grid, 256, 0, s, pdl_enabled(), reinterpret_cast<const uint4*>(x),
               int(T), int(G), int(NG), int(P), int(Ta), reinterpret_cast<uint4*>(xq), (int32_t*)nullptr, sf);
  return cuda_status(e);
}

extern "C" __attribute__((visibility("default"))) fq_status quant_fp8_group_ue8m0_packed(const uint16_t* x, int64_t T, int64_t G, int64_t D,
                                                  uint8_t* xq, int32_t* s_packed, fq_stream_t stream) {
  return fp8_group_common(x, T, G, D, xq, s_packed, nullptr, stream, true);
}

extern "C" __attribute__((visibility("default"))) fq_status quant_fp8_group_fp32(const uint16_t* x, int64_t T, int64_t G, int64_t D, uint8_t* xq,
                                          float* s_f32, fq_stream_t stream) {
  return fp8_group_common(x, T, G, D, xq, nullptr, s_f32, stream, false);
}

extern "C" __attribute__((visibility("default"))) fq_status fq_pack_scales_ue8m0(const float* s_f32, int64_t T, int64_t G, int64_t NG, int32_t* s_packed,
                                          fq_stream_t stream) {
  if (T < 0 || G < 0 || NG < 0 || T > (int64_t(1) << 30) || G > (int64_t(1) << 20) || NG > (int64_t(1) << 20))
    return FQ_ERR_SHAPE;
  const int64_t P = (NG + 3) / 4, Ta = (T + 3) / 4 * 4;
  const int64_t words = G * P * Ta;
  if (words == 0) return FQ_OK;
  if (!s_packed || (!s_f32 && T > 0)) return FQ_ERR_NULL;
  if (!aligned16(s_packed) || (s_f32 && !aligned16(s_f32))) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int grid = grid_for(words, 256, d.sm_count, 8);
  return cuda_status(launch(pack_scales_kernel, grid, 256, 0, reinterpret_cast<cudaStream_t>(stream), pdl_enabled(),
                            s_f32, int(T), int(G), int(NG), int(P), int(Ta), s_packed));
}

extern "C" __attribute__((visibility("default"))) fq_status fq_quantize_weight_fp8_block(const float* w_gnd, int64_t G, int64_t N, int64_t D, uint8_t* wq,
                                                  float* sw_blk, fq_stream_t stream) {
  if (G < 0 || N < 0 || D < 0 || N % 128 || D % 128 || G * (N / 128) * (D / 128) > (int64_t(1) << 31))
    return FQ_ERR_SHAPE;
  const int64_t blocks = G * (N / 128) * (D / 128);
  if (blocks == 0) return FQ_OK;
  if (!w_gnd || !wq || !sw_blk) return FQ_ERR_NULL;
  if (!aligned16(w_gnd) || !aligned16(wq) || !aligned16(sw_blk)) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  return cuda_status(launch(quantize_weight_fp8_kernel, int(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream),
                            false, reinterpret_cast<const float4*>(w_gnd), int(G), int(N), int(D),
                            reinterpret_cast<uint32_t*>(wq), sw_blk));
}

static fq_status rmsnorm_common(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M, int64_t K, void* q,
                                float* sx, int32_t* s_packed, fq_stream_t stream, bool fp8) {
  if (!(eps >= 0.0f) || !(eps <= 3.4e38f)) return FQ_ERR_ARG;  // finite, non-negative
  if (M < 0 || K < 0 || K % (fp8 ? 128 : 16) || K > 16384 || M > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  if (M == 0 || K == 0) return FQ_OK;
  if (!x || !gamma || !q || (fp8 ? !s_packed : !sx)) return FQ_ERR_NULL;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(q) || !aligned16(fp8 ? (const void*)s_packed : (const void*)sx))
    return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int64_t K8 = K / 8;
  const int64_t rows = fp8 ? (M + 3) / 4 * 4 : M;
  const int P = int((K / 128 + 3) / 4), Ta = int((M + 3) / 4 * 4);
  // More CTAs than the SMs hold at once: one row per CTA at a time, so the
  // extra rows in flight pay (a one-wave grid measured 153.4 -> 155.5 us at
  // M=16384, K=4096, on GB300).
  const int grid = grid_for(rows, 1, d.sm_count, 8);
  const int64_t vpt = (K8 + 255) / 256;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = pdl_enabled();
  auto xp = reinterpret_cast<const uint4*>(x);
  auto gp = reinterpret_cast<const uint4*>(gamma);
  auto qp = reinterpret_cast<uint2*>(q);
  cudaError_t e;
#define FQ_RMS_LAUNCH(V)                                                                                          \
  (fp8 ? launch(rmsnorm_quant_kernel<V, true>, grid, 256, 0, s, pdl, xp, gp, eps, rows, M, K8, qp, sx, s_packed, P, \
                Ta)                                                                                                \
       : launch(rmsnorm_quant_kernel<V, false>, grid, 256, 0, s, pdl, xp, gp, eps, rows, M, K8, qp, sx, s_packed,  \
                P, Ta))
  if (vpt <= 1)
    e = FQ_RMS_LAUNCH(1);
  else if (vpt <= 2)
    e = FQ_RMS_LAUNCH(2);
  else if (vpt <= 4)
    e = FQ_RMS_LAUNCH(4);
  else
    e = FQ_RMS_LAUNCH(8);
#undef FQ_RMS_LAUNCH
  return cuda_status(e);
}

extern "C" __attribute__((visibility("default"))) fq_status rmsnorm_quant_int8(const uint16_t* x, const uint16_t* gamma,
                                                                               float eps, int64_t M, int64_t K,
                                                                               int8_t* xq, float* sx,
                                                                               fq_stream_t stream) {
  return rmsnorm_common(x, gamma, eps, M, K, xq, sx, nullptr, stream, false);
}

extern "C" __attribute__((visibility("default"))) fq_status rmsnorm_quant_fp8_ue8m0_packed(
    const uint16_t* x, const uint16_t* gamma, float eps, int64_t T, int64_t K, uint8_t* xq, int32_t* s_packed,
    fq_stream_t stream) {
  return rmsnorm_common(x, gamma, eps, T, K, xq, nullptr, s_packed, stream, true);
}

extern "C" __attribute__((visibility("default"))) fq_status quant_mxfp8(const uint16_t* x, int64_t R, int64_t K,
                                                                        uint8_t* q, uint8_t* sf_blocked,
                                                                        fq_stream_t stream) {
  if (R < 0 || K < 0 || K % 128 || K > (int64_t(1) << 20) || R > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  if (R == 0 || K == 0) return FQ_OK;
  if (!x || !q || !sf_blocked) return FQ_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf_blocked)) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int64_t K8 = K / 8;
  // Four vectors a thread once the work exceeds one per resident thread
  // (GB300, M=16384, K=4096: 45.2 -> 38.4 us); one otherwise, where the
  // empty slots would only add latency (M=4: 3.2 against 3.45 us).
  const int64_t work = R * K8;
  const int occ1 = resident_ctas(reinterpret_cast<const void*>(quant_mxfp8_kernel<1>), 256, 8);
  const bool wide = work > int64_t(occ1) * d.sm_count * 256;
  const int grid = wide ? wave_grid(quant_mxfp8_kernel<4>, 256, work, 256, d.sm_count, 8)
                        : grid_for(work, 256, d.sm_count, occ1);
  auto k = wide ? quant_mxfp8_kernel<4> : quant_mxfp8_kernel<1>;
  return cuda_status(launch(k, grid, 256, 0, reinterpret_cast<cudaStream_t>(stream), pdl_enabled(),
                            reinterpret_cast<const uint4*>(x), R, K8, reinterpret_cast<uint2*>(q), sf_blocked));
}
