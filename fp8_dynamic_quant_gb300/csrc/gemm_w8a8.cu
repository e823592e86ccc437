// W8A8 linear for decode-sized M on sm_103a: dense (w8a8_linear), fused with
// the per-token quant (w8a8_quant_linear) and grouped per expert
// (w8a8_grouped_linear).
//
// What is computed ("DeepSeek-V4 W8A8 performance analysis", section 1):
//   acc[m, n] = sum_k xq[m, k] * W[k, n]        exact int32
//   y[m, n]   = bf16_RN((fp32(acc) * sx[m]) * sw[n])
//
// How (GB300 design, not the pages' Ascend tiling):
//  * Swap-AB: weight rows (output channels) are the MMA "M" side, decode
//    tokens the narrow "N" side, so a tile is 128 channels x MT tokens
//    (MT = 8/16/32/64) and the weight stream is the only large operand.
//  * Engine: sm_103a has no tcgen05 int8 MMA and its legacy int8 mma.sync
//    runs at ~150 TOPS, while f16 mma.sync runs at ~600 TFLOPS.  int8 values
//    are exact in f16 and their products and sums are exact integers in the
//    fp32 accumulator while |partial| < 2^24, so every 8 k-blocks (1024 K,
//    |partial| <= 1024*127*127 < 2^24) the fp32 accumulator is folded into an
//    int32 one: the GEMM stays exact.  int8 -> f16 is a byte permute onto the
//    f16 pattern of 1024 + (q + 128) followed by one f16x2 subtract.
//  * Operand staging: a producer warp streams (16*CW)x128-byte weight boxes
//    and MTx128-byte activation boxes with TMA (cp.async.bulk.tensor,
//    128-byte swizzle) into a multi-stage mbarrier ring; CW consumer warps
//    (8, or 14 for 224-row tiles) each own 16 channels, and one converter
//    warp turns each stage's activations into f16 B fragments once for all
//    of them.  Because the K order inside a sum is free, each lane reads one
//    contiguous 16-byte chunk per row and the same physical-to-logical K
//    permutation is applied to both operands, so no shuffles are needed.
//  * Small N (K=4096, N=1024): 4-CTA clusters split K and reduce through
//    distributed shared memory (with converter warps for token tiles of 32
//    and 64); 32- and 64-token tiles on wide N and the MoE: the tcgen05
//    kernel below.
//  * Scheduling: stream-K.  The (tile, k-block) iteration space is cut into
//    equal contiguous ranges, one per CTA (one CTA per SM), which balances
//    any (M, N, K) across all 152 SMs - the role the pages give to baseM /
//    SmallMN / StreamK tiling ("QuantMatmul small-M tiling", section 3).
//    A CTA's first and last tiles may be partial: their int32 partials go to
//    per-CTA workspace slots, and the last CTA to finish a tile (counted with
//    an atomic per tile) adds them up and runs the dequant epilogue.  Integer
//    sums make the result independent of that order.  When 224-row tiles
//    give 3/4 to 1 tile per SM (up to 16 tokens), each CTA streams one whole
//    tile instead, and the fused op with up to 14 tokens is one launch whose
//    CTAs quantize the activations themselves.
//  * Weights are read with an L2 evict-first hint; activations evict-last.
//  * Programmatic dependent launch: weight loads for the first stages are
//    issued at kernel entry, before griddepcontrol.wait, overlapping the
//    previous kernel - how many, the host picks by what the kernel requests
//    right after the wait.  (Library calls that can write a weight operand
//    let the next kernel start only once they have finished.)
#include <cuda_fp16.h>

#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fq_common.cuh"

namespace fq {

constexpr int kBK = 128;             // K bytes per k-block
constexpr int kFlushBlocks = 8;      // fold fp32 -> int32 every 8 k-blocks (1024 K)
constexpr int kBN = 128;             // weight rows per tile in the stream-K configuration (8 consumer warps)

// Largest K whose whole quantized activation tile a CTA keeps in shared
// memory when it quantizes the activations itself.
constexpr int kFuseKMax = 1024;

// MT tokens per tile, CW consumer warps of 16 weight rows each (BN = 16 * CW
// rows per tile), one producer warp and one activation-converter warp.  FQ:
// the CTA quantizes its activations itself (the stages then hold weights only).
template <int MT, int CW, bool FQ = false>
struct Cfg {
  static constexpr int NT = MT / 8;
  static constexpr int BN = 16 * CW;
  static constexpr int THREADS = (CW + 2) * 32;
  static constexpr int W_BYTES = BN * kBK;
  static constexpr int X_BYTES = MT * kBK;
  static constexpr int STAGE = W_BYTES + (FQ ? 0 : X_BYTES);  // multiple of 1024
  static constexpr int XF = MT * kBK * 2;                     // f16 activation fragments of a stage
  static constexpr int XQ = FQ ? MT * kFuseKMax : 0;          // quantized activation tile, all of K
  // Token tiles of up to 16 store the output straight from the MMA fragments;
  // larger ones stage it in shared memory for 16-byte stores.
  static constexpr bool DIRECT_EPI = MT <= 16;
  static constexpr int EPI = DIRECT_EPI ? 0 : BN * MT * 2;    // bf16 staging
  // Loaded HBM latency is several microseconds, so each SM needs ~200 KB of
  // weights in flight to stream at full rate: fill shared memory up to the
  // opt-in maximum (232448 bytes) less the kernel's static tables.
  static constexpr int SMEM_LIMIT = 232448 - 4160;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - EPI - XQ - 1088) / (STAGE + XF + 24);
  static constexpr int STAGES = STAGES_FIT > 24 ? 24 : STAGES_FIT;
  static constexpr int SLOT = BN * MT;                        // int32 per slot
  static constexpr int SMEM = STAGES * (STAGE + XF) + XQ + EPI + 3 * STAGES * 8 + 64 + 1024;  // + alignment slack
  static_assert(STAGES >= 3, "pipeline too shallow");
  static_assert(SMEM <= SMEM_LIMIT, "shared-memory budget");
};

// Fragment row g (0..7) of a 16-row block reads shared-memory row R(g).  The
// 128-byte TMA swizzle XORs the 16-byte chunk index with (row & 7); with this
// permutation the two rows served in one quarter-warp phase of a 16-byte
// ld.shared (g = 2k, 2k+1) land in different 64-byte halves, so every phase
// touches all 32 banks once.
__device__ __forceinline__ int frag_row(int g) { return (g >> 1) | ((g & 1) << 2); }

// The fields a producer reads before its first weight copies come first, so
// that they share one constant-cache line: each extra line is a miss on the
// path to the first copy.
struct Problem {
  int M, N, K, KB;          // tokens (dense) / rows (grouped), channels, depth, k-blocks
  int m_tiles;              // dense: tiles along M
  int n_tiles;              // tiles along N
  int64_t total;            // dense: total iterations (tiles * KB); grouped: computed on device
  int per_cta;              // dense: iterations per CTA when the split is uniform (host-computed), else 0
  int ahead;                // stages the producer keeps in flight (0: the whole ring)
  int w_reuse;              // weight tiles are read by more than one token tile
  int E;                    // grouped: experts
  int pre_w;                // dense: weight stages issued before the wait on the previous kernel (0: all ahead)
  const float* sx;          // [M] or [R]
  const float* sw;          // [N] or [E, N]
  uint16_t* y;              // [M, N] or [R, N]
  int32_t* slots;           // 2 per CTA
  uint32_t* counters;       // per tile
  uint32_t* err;
  const int32_t* offsets;   // grouped: [E + 1]
  const uint16_t* x16;      // CTA-quantized activations: bf16 [M, K]
  int8_t* xq_out;           // ... optional copy of the quantized activations [M, K]
  float* sx_out;            // ... optional copy of their scales [M]
};
static_assert(offsetof(Problem, sx) <= 56, "producer set-up fields within the first 64 bytes");

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// The same load as an ordinary (non-volatile) asm, so the compiler may issue it
// ahead of the MMAs that precede it.  Its address must come from pin() after
// the mbarrier wait that guards the data: the dependency keeps the load from
// moving above the wait; a consuming volatile MMA keeps it from sinking below
// the stage's release.
__device__ __forceinline__ uint4 lds128_nv(uint32_t addr) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t pin(uint32_t v) {
  asm volatile("" : "+r"(v)::"memory");
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// int8 x4 -> two f16x2: lo = (b0, b1), hi = (b2, b3), exactly.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;                 // q + 128 as an unsigned byte
  uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);   // f16 0x64uu = 1024 + u
  uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 lh = __hsub2(*reinterpret_cast<__half2*>(&l), bias);
  __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&h), bias);
  lo = *reinterpret_cast<uint32_t*>(&lh);
  hi = *reinterpret_cast<uint32_t*>(&hh);
}

__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
  return s == 0 ? v.x : (s == 1 ? v.y : (s == 2 ? v.z : v.w));
}

// Tile -> operand coordinates.
struct TileCoord {
  int w_row;     // first weight row in the (possibly expert-stacked) weight tensor
  int x_row;     // first activation row
  int rows;      // valid activation rows in this tile (<= MT)
  int n0;        // first output channel
  int sw_base;   // offset of this tile's expert in sw
};

template <int MT, int BN, bool GROUPED>
__device__ __forceinline__ TileCoord decode_tile(const Problem& p, int tile, const int* tile_start) {
  TileCoord tc;
  if (!GROUPED) {
    const int mtl = p.m_tiles;
    const int nt = mtl == 1 ? tile : tile / mtl, mt = tile - nt * mtl;
    tc.w_row = nt * BN;
    tc.n0 = nt * BN;
    tc.x_row = mt * MT;
    tc.rows = min(MT, p.M - mt * MT);
    tc.sw_base = 0;
  } else {
    // binary search the expert whose tile range holds `tile`
    int lo = 0, hi = p.E;  // tile_start[lo] <= tile < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_start[mid] <= tile) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int r0 = p.offsets[e], me = p.offsets[e + 1] - r0;
    const int mtn = (me + MT - 1) / MT;
    const int local = tile - tile_start[e];
    const int nt = local / mtn, mt = local % mtn;
    tc.w_row = e * p.N + nt * BN;
    tc.n0 = nt * BN;
    tc.x_row = r0 + mt * MT;
    tc.rows = min(MT, me - mt * MT);
    tc.sw_base = e * p.N;
  }
  return tc;
}

// Stream-K ranges: CTA b owns iterations [rb[b], rb[b+1]) with
// rb[b] = floor(b * I / G), tabulated once per CTA in shared memory.
constexpr int kMaxGrid = 1024;
// CTA whose range holds iteration i: the largest c with rb[c] <= i (rb ascending, rb[0] = 0).
__device__ __forceinline__ int cta_of(const int* rb, int G, int i) {
  int lo = 0, hi = G;  // rb[lo] <= i < rb[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (rb[mid] <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// First iteration of CTA c's range in a dense problem, floor(c * total / G):
// the host passes the per-CTA count when the split is uniform, which keeps the
// 64-bit division off the path to a CTA's first weight copy.
__device__ __forceinline__ int range_begin(const Problem& p, int c, int G) {
  return p.per_cta ? c * p.per_cta : int(int64_t(c) * p.total / G);
}

// ---------------------------------------------------------------- the kernel
template <int MT, int CW, bool GROUPED, bool FQ = false>
__global__ void __launch_bounds__(Cfg<MT, CW, FQ>::THREADS, 1)
    w8a8_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, Problem p) {
  using C = Cfg<MT, CW, FQ>;
  static_assert(!(FQ && GROUPED), "CTA-quantized activations: dense problems only");
  constexpr int NT = C::NT, S = C::STAGES, BN = C::BN, kThreads = C::THREADS, kCW = CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* xfrag = smem + S * C::STAGE;  // [S][h][NT][2][32 lanes] x 16 bytes of f16 B fragments
  // FQ: the quantized activation tile, [k-block][MT rows][128 bytes], 16-byte
  // chunks swizzled like the TMA's 128-byte mode (chunk ^ (row & 7))
  uint8_t* xqs = smem + S * (C::STAGE + C::XF);
  uint16_t* epi = reinterpret_cast<uint16_t*>(smem + S * (C::STAGE + C::XF) + C::XQ);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * (C::STAGE + C::XF) + C::XQ + C::EPI);
  uint64_t* empty = full + S;
  uint64_t* xready = empty + S;
  __shared__ float s_sxq[FQ ? MT : 1];
  __shared__ unsigned s_amax[FQ ? MT : 1];  // FQ: row absmax bits (non-negative floats order as integers)
  __shared__ float s_inv[FQ ? MT : 1];      // FQ: reciprocal of each row's scale
  __shared__ int s_flag;
  __shared__ int s_issued, s_consumed;
  __shared__ volatile int s_abort;  // set after any timed-out wait: later waits are skipped
  __shared__ int tile_start_s[GROUPED ? 1025 : 1];
  __shared__ int rb[kMaxGrid + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const bool producer = warp == kCW && lane == 0;
  if (FQ && tid < MT) s_amax[tid] = 0u;  // before the first block barrier
  constexpr int kConv = CW + 1;  // the activation-converter warp
  // The producer thread sets up the ring and, for dense problems, issues the
  // first stages of weights before anything else: they depend on nothing, and
  // at decode sizes every cycle before the first copy adds to the kernel time.
  int pre = 0;  // weight stages already issued (producer thread)
  if (producer) {
    // the barriers the first copies complete on come first; the rest after
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    if (!GROUPED) {
      // this CTA's stream-K range, as rb[] below tabulates it
      const int b0 = range_begin(p, b, G), b1 = range_begin(p, b + 1, G);
      pre = min(b1 - b0, p.ahead > 0 && p.ahead < S ? p.ahead : S);
      if (p.pre_w > 0 && p.pre_w < pre) pre = p.pre_w;
      const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      // one whole tile per CTA: no division
      int tile = p.per_cta == p.KB ? b : b0 / p.KB, kb = b0 - tile * p.KB;
      TileCoord tc = decode_tile<MT, BN, GROUPED>(p, tile, nullptr);
      for (int r = 0; r < pre; ++r) {
        mbar_arrive_expect_tx(&full[r], C::STAGE);
        tma_load_2d(stages + r * C::STAGE, &tmW, &full[r], kb * kBK, tc.w_row, pol_w);
        if (++kb == p.KB && r + 1 < pre) {
          kb = 0;
          tc = decode_tile<MT, BN, GROUPED>(p, ++tile, nullptr);
        }
      }
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(&empty[i], kCW);
      mbar_init(&xready[i], 1);
    }
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_abort = 0;
    tma_prefetch_desc(&tmX);
  }

  int64_t I = p.total;
  if (GROUPED) {
    // per-expert tile counts from the device offsets (written by moe_sort)
    pdl_wait();
    __shared__ int wsum[kThreads / 32];
    const int NB = p.n_tiles;
    const int per = (p.E + kThreads - 1) / kThreads;
    int local = 0;
    for (int k = 0; k < per; ++k) {
      const int e = tid * per + k;
      if (e < p.E) {
        const int me = p.offsets[e + 1] - p.offsets[e];
        local += me > 0 ? NB * ((me + MT - 1) / MT) : 0;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int k = 0; k < per; ++k) {
      const int e = tid * per + k;
      if (e < p.E) {
        tile_start_s[e] = run;
        const int me = p.offsets[e + 1] - p.offsets[e];
        run += me > 0 ? NB * ((me + MT - 1) / MT) : 0;
      }
    }
    if (tid == kThreads - 1) tile_start_s[p.E] = run;
    __syncthreads();
    I = int64_t(tile_start_s[p.E]) * p.KB;
  }
  __syncthreads();

  for (int c = tid; c <= G; c += kThreads) rb[c] = GROUPED ? int(int64_t(c) * I / G) : range_begin(p, c, G);
  __syncthreads();
  const int begin = rb[b], end = rb[b + 1];
  const int KB = p.KB;

  if (warp == kCW) {
    // ------------------------------------------------ producer warp
    if (lane == 0 && end > begin) {
      // weights streamed once: evict-first; weights shared by several token
      // tiles (large M, big experts) stay in L2 for the next token tile
      const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int n_it = end - begin;
      // stages kept in flight: the whole ring, or fewer so that the first
      // ones land sooner and the consumers start while the rest stream
      const int AH = p.ahead > 0 && p.ahead < S ? p.ahead : S;
      const int npre = n_it < AH ? n_it : AH;
      // weight stages issued at kernel entry (the rest of the first AH go out
      // right after the wait, into ring slots not yet used)
      const int pre_w = (!GROUPED && p.pre_w > 0 && p.pre_w < npre) ? p.pre_w : npre;
      // weights do not depend on the previous kernel: issue them first
      // (dense problems issued them at kernel entry)
      if (GROUPED) {
        int tile = begin / KB, kb = begin - tile * KB;
        TileCoord tc = decode_tile<MT, BN, GROUPED>(p, tile, tile_start_s);
        for (int r = 0; r < npre; ++r) {
          mbar_arrive_expect_tx(&full[r], C::STAGE);
          tma_load_2d(stages + r * C::STAGE, &tmW, &full[r], kb * kBK, tc.w_row, pol_w);
          if (++kb == KB && r + 1 < npre) {
            kb = 0;
            tc = decode_tile<MT, BN, GROUPED>(p, ++tile, tile_start_s);
          }
        }
      }
      pdl_wait();
      int tile = begin / KB, kb = begin - tile * KB;
      TileCoord tc = decode_tile<MT, BN, GROUPED>(p, tile, tile_start_s);
      int issued = 0;
      for (int r = 0; r < n_it; ++r) {
        const int s = r % S;
        if (r < pre_w) {
          if (!FQ) tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], kb * kBK, tc.x_row, pol_x);
        } else if (r < npre) {
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          tma_load_2d(stages + s * C::STAGE, &tmW, &full[s], kb * kBK, tc.w_row, pol_w);
          if (!FQ) tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], kb * kBK, tc.x_row, pol_x);
        } else {
          // iteration r - AH consumed: at most AH stages in flight, and (as
          // r - S <= r - AH) slot s is free
          const int rq = r - AH;
          if (s_abort || !mbar_wait(&empty[rq % S], uint32_t((rq / S) & 1))) {
            if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          tma_load_2d(stages + s * C::STAGE, &tmW, &full[s], kb * kBK, tc.w_row, pol_w);
          if (!FQ) tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], kb * kBK, tc.x_row, pol_x);
        }
        ++issued;
        if (++kb == KB && r + 1 < n_it) {
          kb = 0;
          tc = decode_tile<MT, BN, GROUPED>(p, ++tile, tile_start_s);
        }
      }
      s_issued = issued;
    }
  } else if (warp == kConv) {
    // ------------------------------------------------ activation converter
    // Every consumer warp needs the same f16 B fragments of a stage's
    // activation tile; converting them once here takes that integer work
    // (a third of the consumers' at 8 tokens) off the fourteen consumer
    // warps.  Lane l writes what consumer lane l reads: for each 64-byte half
    // h and token group j, the f16 pairs of its 16-byte chunk, k16 steps 0-1
    // then 2-3.
    const int g = lane >> 2, c = lane & 3;
    const int rg = frag_row(g);
    const uint32_t sbase = smem_u32(stages), xbase = smem_u32(xfrag), xqbase = smem_u32(xqs);
    const int n_it = end - begin;
    // FQ: wait until the consumer warps have quantized the activation tile
    if (FQ) named_bar_sync(2, (kCW + 1) * 32);
    int kb = begin % KB;
    for (int r = 0; r < n_it; ++r) {
      const int s = r % S;
      if (!mbar_wait_try_first(&full[s], uint32_t((r / S) & 1), &s_abort)) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = FQ ? xqbase + uint32_t(kb * MT * kBK) : sbase + uint32_t(s * C::STAGE) + uint32_t(C::W_BYTES);
      if (++kb == KB) kb = 0;
      const uint32_t xo = xbase + uint32_t(s * C::XF);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t q = uint32_t(((4 * h + c) ^ rg) << 4);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint4 v = lds128(st + uint32_t((8 * j + rg) * kBK) + q);
          uint32_t f[8];
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) i8x4_to_f16(word_of(v, ks), f[2 * ks], f[2 * ks + 1]);
          const uint32_t o = xo + uint32_t(((h * NT + j) * 2) * 512 + lane * 16);
          sts128(o, f[0], f[1], f[2], f[3]);
          sts128(o + 512, f[4], f[5], f[6], f[7]);
        }
      }
      // generic-proxy reads of the stage before the async-proxy refill
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&xready[s]);
    }
  } else {
    // ------------------------------------------------ consumer warps
    pdl_wait();
    // Let the next kernel launch only once this one's inputs are final: a
    // dependent may prefetch weights before its own wait, which is safe only
    // if every earlier kernel has finished.
    pdl_launch_dependents();
    if constexpr (FQ) {
      // Per-token quant of the whole activation tile (one tile per CTA, all of
      // K) with the quant kernel's arithmetic; the row max does not depend on
      // the order, so the scale and codes are the quant kernel's bit for bit.
      // CTA 0 also writes the optional copies.  Meanwhile the first weight
      // stages are in flight.
      const int rows = min(MT, p.M);
      const int K8 = p.K / 8;
      const uint32_t xqbase = smem_u32(xqs);
      if (rows <= 4) {
        // Few rows: all consumer threads share the tile.  Thread t takes the
        // 16-byte vectors t, t + kCW * 32, ... of the rows x K/8 vectors;
        // each warp reduces the row maxima of its 32 consecutive vectors and
        // posts them with a shared atomicMax on the float bits (non-negative:
        // a NaN vector counts as 0, as fmaxf ignores it).  GB300, K=1024,
        // N=32768: M = 1 / 4 8.1 -> 7.9 / 8.8 -> 8.5 us against one row per
        // warp; from 7 rows on the two consumer barriers cost more than that
        // saves.
        const int nvec = rows * K8;
        constexpr int kCT = kCW * 32;                              // consumer threads
        constexpr int NV = (4 * (kFuseKMax / 8) + kCT - 1) / kCT;  // vectors per thread, at most (rows <= 4)
        const uint4* xv = reinterpret_cast<const uint4*>(p.x16);   // rows of K8 vectors, contiguous
        uint4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int e = tid + i * kCT;
          if (e < nvec) v[i] = ld_stream(xv + e);
        }
        float a[NV];
        int row[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int e = tid + i * kCT;
          a[i] = e < nvec ? fmaxf(0.0f, absmax8_bf16(v[i])) : 0.0f;
          row[i] = (e < nvec ? e : nvec - 1) / K8;
        }
        if (K8 % 32 == 0) {
          // a warp's 32 vectors lie in one row: a butterfly max, the chains interleaved
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) a[i] = fmaxf(a[i], __shfl_xor_sync(0xFFFFFFFFu, a[i], o));
#pragma unroll
          for (int i = 0; i < NV; ++i)
            if (lane == 0 && i * kCT + warp * 32 < nvec) atomicMax(&s_amax[row[i]], __float_as_uint(a[i]));
        } else {
          // rows shorter than a warp's vectors, or not aligned to them: segmented max
#pragma unroll
          for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              const float ao = __shfl_down_sync(0xFFFFFFFFu, a[i], o);
              const int ro = __shfl_down_sync(0xFFFFFFFFu, row[i], o);
              if (lane + o < 32 && ro == row[i]) a[i] = fmaxf(a[i], ao);
            }
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            const int rprev = __shfl_up_sync(0xFFFFFFFFu, row[i], 1);
            if (tid + i * kCT < nvec && (lane == 0 || rprev != row[i])) atomicMax(&s_amax[row[i]], __float_as_uint(a[i]));
          }
        }
        named_bar_sync(3, kCT);
        if (tid < rows) {
          const float sc = __fdiv_rn(__uint_as_float(s_amax[tid]), 127.0f);
          s_sxq[tid] = sc;
          s_inv[tid] = __frcp_rn(sc);
          if (b == 0 && p.sx_out) p.sx_out[tid] = sc;
        }
        named_bar_sync(3, kCT);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const int e = tid + i * kCT;
          if (e < nvec) {
            const int m = row[i], idx = e - m * K8;
            float f[8];
            unpack8(v[i], f);
            const uint2 qv = quant8_i8(f, s_sxq[m], s_inv[m]);
            const int k = idx * 8;
            const uint32_t sa = xqbase + uint32_t(((k >> 7) * MT + m) * kBK + ((((k >> 4) & 7) ^ (m & 7)) << 4) + (k & 8));
            asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(sa), "r"(qv.x), "r"(qv.y) : "memory");
            if (b == 0 && p.xq_out) *reinterpret_cast<uint2*>(p.xq_out + int64_t(m) * p.K + k) = qv;
          }
        }
      } else {
        // One row per warp (rows m = warp, warp + kCW, ...; a warp's loads
        // issued before its reductions).
        constexpr int VPL = kFuseKMax / 256;       // 16-byte vectors per lane
        constexpr int RPW = (MT + kCW - 1) / kCW;  // rows per warp
        uint4 v[RPW][VPL];
        float amax[RPW];
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
          const int m = warp + u * kCW;
          const uint4* xr = reinterpret_cast<const uint4*>(p.x16) + int64_t(m) * K8;
          amax[u] = 0.0f;
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            const int idx = lane + 32 * i;
            if (m < rows && idx < K8) {
              v[u][i] = ld_stream(xr + idx);
              amax[u] = fmaxf(amax[u], absmax8_bf16(v[u][i]));
            }
          }
        }
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
          const int m = warp + u * kCW;
          if (m >= rows) break;  // warp-uniform
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax[u] = fmaxf(amax[u], __shfl_xor_sync(0xFFFFFFFFu, amax[u], o));
          const float sc = __fdiv_rn(amax[u], 127.0f);
          const float inv = __frcp_rn(sc);
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            const int idx = lane + 32 * i;
            if (idx < K8) {
              float f[8];
              unpack8(v[u][i], f);
              const uint2 qv = quant8_i8(f, sc, inv);
              const int k = idx * 8;
              const uint32_t sa = xqbase + uint32_t(((k >> 7) * MT + m) * kBK + ((((k >> 4) & 7) ^ (m & 7)) << 4) + (k & 8));
              asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(sa), "r"(qv.x), "r"(qv.y) : "memory");
              if (b == 0 && p.xq_out) *reinterpret_cast<uint2*>(p.xq_out + int64_t(m) * p.K + k) = qv;
            }
          }
          if (lane == 0) {
            s_sxq[m] = sc;
            if (b == 0 && p.sx_out) p.sx_out[m] = sc;
          }
        }
      }
      named_bar_sync(2, (kCW + 1) * 32);  // with the converter warp
    }
    const int g = lane >> 2, c = lane & 3;
    const int rg = frag_row(g);
    // With few token tiles, two fp32 chains (even / odd 64-byte halves of a
    // k-block) halve the dependent-MMA latency; both fold into the exact int32
    // sum.  With NT >= 4 the token tiles already give independent chains.
    constexpr int NACC = NT <= 2 ? 2 : 1;
    float accf[NACC][NT][4];
    int acci[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int a = 0; a < NACC; ++a) accf[a][j][r] = 0.f;
        acci[j][r] = 0;
      }
    const uint32_t sbase = smem_u32(stages), xbase = smem_u32(xfrag);
    const uint32_t rowW0 = uint32_t((16 * warp + rg) * kBK), rowW1 = rowW0 + 8 * kBK;
    int tile = begin / KB, kb = begin - tile * KB;
    int seg_kb0 = kb;
    int nk = 0;
    bool first_seg = true;
    int consumed = 0;
    const int n_it = end - begin;
    // Dequant scales of the current tile, loaded when its segment starts so the
    // epilogue does not wait on a global round trip.
    float sxr[NT][2], swr[2];
    int rows_cur = MT;  // valid activation rows of the current tile
    auto load_scales = [&](int t) {
      const TileCoord tc = decode_tile<MT, BN, GROUPED>(p, t, tile_start_s);
      rows_cur = tc.rows;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ml = 8 * j + frag_row(2 * c + h);
          sxr[j][h] = ml < tc.rows ? (FQ ? s_sxq[ml] : __ldg(p.sx + tc.x_row + ml)) : 0.f;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = tc.n0 + 16 * warp + rg + 8 * h;
        swr[h] = n < p.N ? __ldg(p.sw + tc.sw_base + n) : 0.f;
      }
    };
    if (n_it > 0) load_scales(tile);
    // After a timeout (s_abort) the loop keeps its shape - same segments, same
    // named barriers - but skips waits and math, so every warp finishes.
    for (int r = 0; r < n_it; ++r) {
      const int s = r % S;
      const uint32_t par = uint32_t((r / S) & 1);
      bool ok = mbar_wait_try_first(&full[s], par, &s_abort) && mbar_wait_try_first(&xready[s], par, &s_abort);
      if (!ok) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
      }
      const uint32_t st = pin(sbase + uint32_t(s * C::STAGE));
      const uint32_t xo = pin(xbase + uint32_t(s * C::XF) + uint32_t(lane * 16));
#pragma unroll
      for (int h = 0; h < 2 && ok; ++h) {
        const uint32_t q = uint32_t(((4 * h + c) ^ rg) << 4);
        const uint4 wa = lds128_nv(st + rowW0 + q);
        const uint4 wb = lds128_nv(st + rowW1 + q);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // B fragments of k16 steps 2*half and 2*half+1; 8-token groups past
          // the tile's valid rows are skipped (uniform branch): an expert with
          // 3 tokens in a 64-token tile costs one group
          uint4 xv[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j)
            if (8 * j < rows_cur) xv[j] = lds128_nv(xo + uint32_t(((h * NT + j) * 2 + half) * 512));
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int ks = 2 * half + kk;
            uint32_t a0, a1, a2, a3;
            i8x4_to_f16(word_of(wa, ks), a0, a2);
            i8x4_to_f16(word_of(wb, ks), a1, a3);
#pragma unroll
            for (int j = 0; j < NT; ++j)
              if (8 * j < rows_cur)
                mma_f16(accf[h % NACC][j], a0, a1, a2, a3, word_of(xv[j], 2 * kk), word_of(xv[j], 2 * kk + 1));
          }
        }
      }
      // The stage was read through the generic proxy (ld.shared); the next
      // TMA write into it goes through the async proxy.  Order the two before
      // handing the stage back, or TMA can overwrite it under the read.
      fence_proxy_async_smem();
      __syncwarp();
      if (ok) {
        if (lane == 0) mbar_arrive(&empty[s]);
        ++consumed;
      }
      const bool seg_end = (kb == KB - 1) || (r == n_it - 1);
      if (++nk == kFlushBlocks || seg_end) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
              acci[j][rr] += __float2int_rn(accf[a][j][rr]);
              accf[a][j][rr] = 0.f;
            }
          }
        nk = 0;
      }
      if (seg_end) {
        // ---- segment end: tile `tile`, k-blocks [seg_kb0, kb]
        const TileCoord tc = decode_tile<MT, BN, GROUPED>(p, tile, tile_start_s);
        const bool whole = (seg_kb0 == 0) && (kb == KB - 1);
        bool do_epi = whole;
        if (!whole) {
          int32_t* my = p.slots + (2 * b + (first_seg ? 0 : 1)) * int64_t(C::SLOT);
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) my[((warp * NT + j) * 4 + rr) * 32 + lane] = acci[j][rr];
          named_bar_sync(1, kCW * 32);
          if (tid == 0) {
            const uint32_t nb = uint32_t(kb - seg_kb0 + 1);
            const uint32_t old = atom_add_acq_rel_gpu(&p.counters[tile], nb);
            const int last = (old + nb == uint32_t(KB)) ? 1 : 0;
            if (last) p.counters[tile] = 0;  // every contributor has arrived; ready for the next call
            s_flag = last;
          }
          named_bar_sync(1, kCW * 32);
          do_epi = s_flag != 0;
          if (do_epi) {
            // add the other contributors' partials; U slots in flight at once
            constexpr int U = NT <= 2 ? 8 : (NT <= 4 && CW <= 8 ? 4 : 1);
            const int c0 = cta_of(rb, G, tile * KB), c1 = cta_of(rb, G, tile * KB + KB - 1);
            for (int cb = c0; cb <= c1; cb += U) {
              int32_t v[U][NT][4];
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int cc = cb + u;
                // skip self and CTAs with an empty range (more CTAs than iterations)
                const bool use = cc <= c1 && cc != b && rb[cc + 1] != rb[cc];
                const int first_tile = use ? rb[cc] / KB : 0;
                const int32_t* sl = p.slots + (2 * int64_t(cc) + (first_tile == tile ? 0 : 1)) * int64_t(C::SLOT);
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                  for (int rr = 0; rr < 4; ++rr)
                    v[u][j][rr] = use ? __ldcg(sl + ((warp * NT + j) * 4 + rr) * 32 + lane) : 0;
              }
#pragma unroll
              for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                  for (int rr = 0; rr < 4; ++rr) acci[j][rr] += v[u][j][rr];
            }
          }
        }
        if (do_epi && C::DIRECT_EPI) {
          // Dequant and store straight from the fragments: channels rg and
          // rg ^ 1 of a 16-row block sit in lanes l and l ^ 8 (g ^ 2), so the
          // lane holding the even channel stores the pair as one bf16x2 word
          // (N is a multiple of 16: the odd channel is in range with the even).
          const bool lead = (g & 2) == 0;
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int nl = 16 * warp + rg + ((rr & 2) ? 8 : 0);
              const int ml = 8 * j + frag_row(2 * c + (rr & 1));
              const int n = tc.n0 + nl;
              const bool in = ml < tc.rows && n < p.N;
              float v = 0.f;
              if (in) v = __fmul_rn(__fmul_rn(__int2float_rn(acci[j][rr]), sxr[j][rr & 1]), swr[rr >> 1]);
              const uint32_t mine = f32_to_bf16_bits(v);
              const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, mine, 8);
              if (lead && in) *reinterpret_cast<uint32_t*>(p.y + int64_t(tc.x_row + ml) * p.N + n) = mine | (other << 16);
            }
        } else if (do_epi) {
          // dequant into the bf16 staging tile epi[m][n], then coalesced stores
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int nl = 16 * warp + rg + ((rr & 2) ? 8 : 0);
              const int ml = 8 * j + frag_row(2 * c + (rr & 1));
              const int n = tc.n0 + nl;
              float v = 0.f;
              if (ml < tc.rows && n < p.N)
                v = __fmul_rn(__fmul_rn(__int2float_rn(acci[j][rr]), sxr[j][rr & 1]), swr[rr >> 1]);
              epi[ml * BN + nl] = f32_to_bf16_bits(v);
            }
          named_bar_sync(1, kCW * 32);
          for (int idx = tid; idx < MT * (BN / 8); idx += kCW * 32) {
            const int ml = idx / (BN / 8), c8 = idx % (BN / 8);
            const int n = tc.n0 + c8 * 8;
            if (ml < tc.rows && n < p.N) {
              const uint4 v = *reinterpret_cast<const uint4*>(epi + ml * BN + c8 * 8);
              *reinterpret_cast<uint4*>(p.y + int64_t(tc.x_row + ml) * p.N + n) = v;
            }
          }
          named_bar_sync(1, kCW * 32);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) acci[j][rr] = 0;
        first_seg = false;
        seg_kb0 = 0;
      }
      if (++kb == KB) {
        kb = 0;
        ++tile;
        if (r + 1 < n_it) load_scales(tile);
      }
    }
    if (tid == 0) s_consumed = consumed;
  }
  __syncthreads();
  // Drain: on the normal path every issued stage was consumed.  After a
  // timeout, wait (bounded) for copies still in flight before exiting.
  if (tid == 0) {
    for (int r = s_consumed; r < s_issued; ++r) mbar_wait(&full[r % S], uint32_t((r / S) & 1));
  }
}

// ---------------------------------------------------------------- cluster split-K
//
// For problems with too few weight tiles to fill the GPU (e.g. N = 1024), a
// cluster of CL CTAs shares one tile of BN = 8 * CL weight rows and splits K.
// Each CTA accumulates its K-range exactly (int32), then the partials are
// reduce-scattered through distributed shared memory: CTA q of the cluster
// owns rows [8q, 8q + 8) of the tile, receives the partial slices of those
// rows, sums them, dequantizes and writes 16-byte rows of y.  No global
// partial sums, counters or second pass.
// Inside a CTA, KS consumer warps share each 16-row block and split every
// k-block's eight k16 steps among themselves: with one block of rows per
// warp the steps of a k-block form one dependent chain per warp and the
// few warps of a CTA leave the schedulers idle.  Each k-split warp sends
// its own partial slice, so the owner sums CL * KS slices.
template <int MT, int RB, int CL, int KS>
struct CCfg {
  static constexpr int NT = MT / 8;
  static constexpr int BN = 16 * RB;               // RB blocks of 16 weight rows
  static constexpr int CW = RB * KS;               // consumer warps
  // Token tiles of 32 and more: converter warps turn each stage's int8
  // activations into f16 B fragments once (the 224-row kernel's layout), in
  // place of every consumer widening the fragments of its k-split itself -
  // RB times over, on its MMA chain (measured with that widening removed:
  // K=4096, N=1024, M=32 6.0 -> 5.2 us, M=64 8.9 -> 7.0).
  static constexpr bool CONV = MT >= 32;
  static constexpr int XW = CONV ? 4 : 0;  // converter warps, each taking every fourth (half, token group)
  static constexpr int THREADS = (CW + 1 + XW) * 32;
  static constexpr int W_BYTES = BN * kBK;
  static constexpr int X_BYTES = MT * kBK;
  static constexpr int STAGE = W_BYTES + X_BYTES;
  static constexpr int XF = CONV ? MT * kBK * 2 : 0;  // f16 fragments of a stage
  static constexpr int RECV = CL * KS * 8 * MT * 4;  // [CL ranks][KS k-splits][8 rows][MT tokens] int32
  // Token tiles of up to 16: at most ~100 KB, so that two CTAs fit on an SM
  // (with at most 113 registers a thread) and a call's CTAs can start - and
  // stream their weights before their wait on the previous kernel - while
  // the previous call's CTAs still run (K=4096, N=1024, M <= 8: 4.4 -> 4.1
  // us).  Larger tiles keep one CTA per SM and the deeper ring (at 64 tokens
  // the two-per-SM form measured 10.6 against 9.2 us).
  static constexpr int MINB = MT <= 16 ? 2 : 1;
  static constexpr int STAGES_FIT = ((MINB == 2 ? 100 : 212) * 1024 - RECV - 2048) / (STAGE + XF);
  static constexpr int STAGES = STAGES_FIT > (MINB == 2 ? 12 : 16) ? (MINB == 2 ? 12 : 16) : STAGES_FIT;
  static constexpr int SMEM = STAGES * (STAGE + XF) + RECV + 3 * STAGES * 8 + 64 + 1024;
  static_assert(BN == 8 * CL, "each cluster rank owns 8 rows");
  static_assert(KS == 1 || KS == 2 || KS == 4, "k16 steps of a k-block per warp: 8, 4 or 2");
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(!CONV || KS >= 2, "with the converter a warp takes one or both 16-byte fragment pieces of a half");
};

template <int MT, int RB, int CL, int KS>
__global__ void __launch_bounds__(CCfg<MT, RB, CL, KS>::THREADS, CCfg<MT, RB, CL, KS>::MINB)
    w8a8_cluster_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, Problem p) {
  using C = CCfg<MT, RB, CL, KS>;
  constexpr int NT = C::NT, S = C::STAGES, BN = C::BN, kCW = C::CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* xfrag = smem + S * C::STAGE;  // CONV: [S][h][NT][2][32 lanes] x 16 bytes of f16 B fragments
  int32_t* recv = reinterpret_cast<int32_t*>(xfrag + S * C::XF);
  uint64_t* full = reinterpret_cast<uint64_t*>(xfrag + S * C::XF + C::RECV);
  uint64_t* empty = full + S;
  uint64_t* xready = empty + S;  // CONV: the stage's fragments are written
  __shared__ int s_issued, s_consumed;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = int(cluster_ctarank());
  const int tile = blockIdx.x / CL;
  const int KB = p.KB;
  const int kb0 = rank * KB / CL, kb1 = (rank + 1) * KB / CL;
  const int n_it = kb1 - kb0;
  const int npre = n_it < S ? n_it : S;
  const TileCoord tc = decode_tile<MT, BN, false>(p, tile, nullptr);
  // The producer thread sets up the ring and issues the first stages of
  // weights before anything else: they depend on nothing, and at decode sizes
  // every cycle before the first copy adds to the kernel time.
  if (warp == kCW && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
      if (C::CONV) mbar_init(&xready[i], C::XW);
    }
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_abort = 0;
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
    for (int r = 0; r < npre; ++r) {
      mbar_arrive_expect_tx(&full[r], C::STAGE);
      tma_load_2d(stages + r * C::STAGE, &tmW, &full[r], (kb0 + r) * kBK, tc.w_row, pol_w);
    }
  }
  // the ring is initialised before any thread waits on it
  __syncthreads();
  // Every CTA of the cluster must be running before any distributed-smem
  // write: arrive now, wait just before the scatter (keeps it off the
  // critical path of the weight stream).
  cluster_arrive_relaxed();
  // epilogue scales of the rows this CTA owns (8 channels, one token per thread)
  const int n_first = tc.n0 + 8 * rank;
  float sw_own[8];
  float sx_own = 0.f;
#pragma unroll
  for (int r2 = 0; r2 < 8; ++r2) sw_own[r2] = (n_first < p.N) ? __ldg(p.sw + tc.sw_base + n_first + r2) : 0.f;

  if (warp == kCW) {
    if (lane == 0 && n_it > 0) {
      const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      pdl_wait();
      int issued = 0;
      for (int r = 0; r < n_it; ++r) {
        const int s = r % S;
        if (r < npre) {
          tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], (kb0 + r) * kBK, tc.x_row, pol_x);
        } else {
          if (s_abort || !mbar_wait(&empty[s], uint32_t((r / S - 1) & 1))) {
            if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          tma_load_2d(stages + s * C::STAGE, &tmW, &full[s], (kb0 + r) * kBK, tc.w_row, pol_w);
          tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], (kb0 + r) * kBK, tc.x_row, pol_x);
        }
        ++issued;
      }
      s_issued = issued;
    }
    __syncwarp();
    cluster_wait_acquire();  // matches the consumers' wait before their scatter
  } else if (C::CONV && warp > kCW) {
    // ------------------------------------------------ activation converters
    // Converter warp cw takes the (half h, token group j) tasks t = h * NT + j
    // with t % XW == cw.  Lane l converts what consumer lane l reads: the f16
    // pairs of its 16-byte chunk, words 0-1 into one 512-byte piece and words
    // 2-3 into the next.  Rows past M were filled with zeros by the copy.
    const int cw = warp - kCW - 1;
    const int g = lane >> 2, c = lane & 3;
    const int rg = frag_row(g);
    const uint32_t sbase = smem_u32(stages), xbase = smem_u32(xfrag);
    for (int r = 0; r < n_it; ++r) {
      const int s = r % S;
      if (!mbar_wait_try_first(&full[s], uint32_t((r / S) & 1), &s_abort)) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = sbase + uint32_t(s * C::STAGE + C::W_BYTES);
      const uint32_t xo = xbase + uint32_t(s * C::XF) + uint32_t(lane * 16);
      constexpr int XW = C::XW > 0 ? C::XW : 1;  // (the branch is compiled for every MT)
      static_assert(!C::CONV || (2 * NT) % XW == 0, "whole tasks per converter warp");
      uint4 v[2 * NT / XW];
#pragma unroll
      for (int i = 0; i < 2 * NT / XW; ++i) {
        const int t = cw + i * XW, h = t / NT, j = t % NT;
        v[i] = lds128(st + uint32_t((8 * j + rg) * kBK) + uint32_t(((4 * h + c) ^ rg) << 4));
      }
#pragma unroll
      for (int i = 0; i < 2 * NT / XW; ++i) {
        const int t = cw + i * XW;
        uint32_t f[8];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) i8x4_to_f16(word_of(v[i], ks), f[2 * ks], f[2 * ks + 1]);
        const uint32_t o = xo + uint32_t(t * 2 * 512);
        sts128(o, f[0], f[1], f[2], f[3]);
        sts128(o + 512, f[4], f[5], f[6], f[7]);
      }
      // generic-proxy reads of the stage before the async-proxy refill
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&xready[s]);
    }
    __syncwarp();
    cluster_wait_acquire();  // matches the consumers' wait before their scatter
  } else {
    pdl_wait();
    pdl_launch_dependents();
    const int g = lane >> 2, c = lane & 3;
    const int rg = frag_row(g);
    // warp -> (16-row block rbk, k-split kq): kq takes 16-byte chunk half
    // HQ of every k-block row (KS >= 2) and, with KS = 4, two of its four words
    const int rbk = warp % RB, kq = warp / RB;
    constexpr int NH = KS == 1 ? 2 : 1;   // 64-byte halves of a k-block per warp
    constexpr int NW = KS == 4 ? 2 : 4;   // k16 steps per half
    const int h0 = KS == 1 ? 0 : (KS == 2 ? kq : kq >> 1);
    const bool hi_words = KS == 4 && (kq & 1);
    constexpr int NACC = NT <= 2 ? 2 : 1;
    float accf[NACC][NT][4];
    int acci[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int a = 0; a < NACC; ++a) accf[a][j][r] = 0.f;
        acci[j][r] = 0;
      }
    const uint32_t sbase = smem_u32(stages), xbase = smem_u32(xfrag);
    const uint32_t rowW0 = uint32_t((16 * rbk + rg) * kBK), rowW1 = rowW0 + 8 * kBK;
    const int rows_cur = tc.rows;
    int nk = 0, consumed = 0;
    // the four words of a 16-byte chunk, or the two this warp takes
    auto pick = [&](const uint4& v, uint32_t (&w)[NW]) {
      if constexpr (NW == 4) {
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
      } else {
        w[0] = hi_words ? v.z : v.x;
        w[1] = hi_words ? v.w : v.y;
      }
    };
    for (int r = 0; r < n_it; ++r) {
      const int s = r % S;
      const uint32_t par = uint32_t((r / S) & 1);
      bool ok = mbar_wait_try_first(&full[s], par, &s_abort) &&
                (!C::CONV || mbar_wait_try_first(&xready[s], par, &s_abort));
      if (!ok) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
      }
      const uint32_t st = sbase + uint32_t(s * C::STAGE);
      const uint32_t xo = xbase + uint32_t(s * C::XF) + uint32_t(lane * 16);
#pragma unroll
      for (int hh = 0; hh < NH && ok; ++hh) {
        const int h = h0 + hh;
        const uint32_t q = uint32_t(((4 * h + c) ^ rg) << 4);
        uint32_t wa[NW], wb[NW], wx[C::CONV ? 1 : NT][NW];
        uint4 bx[C::CONV ? NT : 1][NW / 2];  // CONV: the fragment pieces of this warp's words
        pick(lds128(st + rowW0 + q), wa);
        pick(lds128(st + rowW1 + q), wb);
        if constexpr (C::CONV) {
          // words 0-1 of the chunk are piece 0, words 2-3 piece 1
#pragma unroll
          for (int j = 0; j < NT; ++j)
            if (8 * j < rows_cur)
#pragma unroll
              for (int pc = 0; pc < NW / 2; ++pc)
                bx[j][pc] = lds128(xo + uint32_t(((h * NT + j) * 2 + (NW == 4 ? pc : (hi_words ? 1 : 0))) * 512));
        } else {
#pragma unroll
          for (int j = 0; j < NT; ++j) pick(lds128(st + C::W_BYTES + uint32_t((8 * j + rg) * kBK) + q), wx[j]);
        }
#pragma unroll
        for (int ks = 0; ks < NW; ++ks) {
          uint32_t a0, a1, a2, a3;
          i8x4_to_f16(wa[ks], a0, a2);
          i8x4_to_f16(wb[ks], a1, a3);
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (8 * j < rows_cur) {
              uint32_t b0, b1;
              if constexpr (C::CONV) {
                const uint4& v = bx[j][NW == 4 ? (ks >> 1) : 0];
                b0 = word_of(v, 2 * (ks & 1));
                b1 = word_of(v, 2 * (ks & 1) + 1);
              } else {
                i8x4_to_f16(wx[j][ks], b0, b1);
              }
              mma_f16(accf[(NH == 2 ? hh : ks) % NACC][j], a0, a1, a2, a3, b0, b1);
            }
          }
        }
      }
      // generic-proxy reads of the stage before the async-proxy refill
      fence_proxy_async_smem();
      __syncwarp();
      if (ok) {
        if (lane == 0) mbar_arrive(&empty[s]);
        ++consumed;
      }
      if (++nk == kFlushBlocks || r == n_it - 1) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int a = 0; a < NACC; ++a) {
              acci[j][rr] += __float2int_rn(accf[a][j][rr]);
              accf[a][j][rr] = 0.f;
            }
        nk = 0;
      }
    }
    if (tid < MT && tid < tc.rows) sx_own = __ldg(p.sx + tc.x_row + tid);
    // reduce-scatter: row 16*rbk + R(g) (+8) belongs to cluster rank 2*rbk (+1);
    // each (rank, k-split) pair has its own slice at the owner
    cluster_wait_acquire();  // all CTAs of the cluster have started
    const uint32_t recv_base = smem_u32(recv);
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int owner = 2 * rbk + (rr >> 1);
        const int ml = 8 * j + frag_row(2 * c + (rr & 1));
        const uint32_t off = uint32_t((((rank * KS + kq) * 8 + rg) * MT + ml) * 4);
        st_cluster_u32(mapa_shared(recv_base + off, uint32_t(owner)), uint32_t(acci[j][rr]));
      }
    if (tid == 0) s_consumed = consumed;
  }
  // all partial slices have landed in their owners' shared memory
  __syncwarp();
  cluster_sync_all();
  if (warp < kCW) {
    // owner epilogue: rows [8 * rank, 8 * rank + 8) of the tile, one token per thread
    for (int ml = tid; ml < MT; ml += kCW * 32) {  // MT <= 64 <= consumer threads: one pass
      if (ml < tc.rows && n_first < p.N) {
        const float sxv = sx_own;
        uint32_t packed[4];
#pragma unroll
        for (int r2 = 0; r2 < 8; r2 += 2) {
          int a0 = 0, a1 = 0;
#pragma unroll
          for (int rk = 0; rk < CL * KS; ++rk) {
            a0 += recv[(rk * 8 + r2) * MT + ml];
            a1 += recv[(rk * 8 + r2 + 1) * MT + ml];
          }
          const float v0 = __fmul_rn(__fmul_rn(__int2float_rn(a0), sxv), sw_own[r2]);
          const float v1 = __fmul_rn(__fmul_rn(__int2float_rn(a1), sxv), sw_own[r2 + 1]);
          packed[r2 / 2] = uint32_t(f32_to_bf16_bits(v0)) | (uint32_t(f32_to_bf16_bits(v1)) << 16);
        }
        *reinterpret_cast<uint4*>(p.y + int64_t(tc.x_row + ml) * p.N + n_first) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    for (int r = s_consumed; r < s_issued; ++r) mbar_wait(&full[r % S], uint32_t((r / S) & 1));
  }
}

// ---------------------------------------------------------------- tcgen05 path (token tiles of 32 / 64)
//
// With 32 or more tokens per tile the mma.sync path above is bound by its own
// instruction stream (the tensor pipe sits at a quarter of its time).  Here
// the 5th-generation tensor cores take the MMA, with the weights as the A
// operand in tensor memory and fp32 accumulators in tensor memory:
//  - warp 0, lane 0: TMA producer of raw int8 stages (128 weight rows x 128 K
//    and MT tokens x 128 K), the same stream-K walk as the kernel above;
//  - warps 2..9: converters, two groups of four taking alternate k-blocks.
//    Warp w reaches tensor-memory lanes 32*(w%4)..32*(w%4)+31: every thread
//    turns the 128 bytes of its weight row into f16 pairs and stores them to
//    the k-block's A stage with tcgen05.st.  Together a group converts the
//    activation tile into a 128-byte-swizzled K-major f16 operand in shared
//    memory.
//  - warp 1: allocates tensor memory; the whole warp walks the k-blocks and
//    an elected lane issues tcgen05.mma kind::f16 (M = 128 weight rows,
//    N = MT tokens, K = 16) and commits each stage back.
//  - warps 10..13: epilogue, one weight row per thread.  They drain each
//    finished accumulator region into exact int32 sums kept in tensor memory
//    and, at a segment's end, run the stream-K hand-off and the dequantizing
//    store - while the converters and the tensor cores go on with the next
//    segment.
// Exactness: an int8 x int8 product is exact in fp32 and 1024 of them sum
// below 2^24, so every 1024-K chunk accumulates in a fresh tensor-memory
// region (two regions alternate) and is rounded to int32 (exact) on the way
// out.
namespace um {
constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kConvWarps + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;

// Tensor-memory columns: [2 buffers] fp32 accumulator regions of MT columns
// (one chain: the K steps of a chunk accumulate into one region - measured as
// fast as four independent chains), then OP_STAGES A stages of 64 columns,
// then MT columns of int32 segment sums.  The A stages pace the pipeline
// (converters -> MMA -> stage released): 5 at 64 tokens and 6 at 32, against
// 3 and 4 with the four-chain layout, took K=1024, N=32768, M=64 from 12.6 to
// 12.2 us and M=32 from 11.6 to 10.8 us on GB300.
template <int MT>
struct Cfg {
  static constexpr int CH = 1;
  static constexpr int ACC_COLS = 2 * CH * MT;
  static constexpr int OP_FIT = (int(kTmemCols) - ACC_COLS - MT) / 64;
  static constexpr int OP_STAGES = OP_FIT > 6 ? 6 : OP_FIT;
  static constexpr int ISUM_COL = ACC_COLS + OP_STAGES * 64;
  static constexpr int W_BYTES = 128 * kBK;       // raw weights of a stage
  static constexpr int X_BYTES = MT * kBK;        // raw activations of a stage
  static constexpr int RAW = W_BYTES + X_BYTES;   // multiple of 1024
  static constexpr int XF = MT * kBK * 2;         // f16 activations: two 64-K halves of MT rows x 128 B
  static constexpr int SMEM_BUDGET = 216 * 1024;
  static constexpr int RAW_FIT = (SMEM_BUDGET - OP_STAGES * XF - 2048) / RAW;
  static constexpr int RAW_STAGES = RAW_FIT > 12 ? 12 : RAW_FIT;
  static constexpr int SLOT = 128 * MT;           // int32 per partial-sum slot
  static constexpr int BAR_BYTES = (2 * RAW_STAGES + 2 * OP_STAGES + 4 + 1) * 8;
  static constexpr int SMEM = RAW_STAGES * RAW + OP_STAGES * XF + BAR_BYTES + 1024;
  static_assert(OP_STAGES >= 2, "operand pipeline too shallow");
  static_assert(ISUM_COL + MT <= int(kTmemCols), "tensor-memory budget");
  static_assert(RAW_STAGES >= 3, "pipeline too shallow");
  static_assert(MT == 32 || MT == 64, "token tile");
};

// Activation box height: only as many token rows as the tile holds (16, 32
// or MT); rows past them in the stage are stale and feed output columns that
// are never stored.
template <int MT>
__device__ __forceinline__ int x_box_rows(int rows) { return rows <= 16 ? 16 : (rows <= 32 ? 32 : MT); }
}  // namespace um


template <int MT, bool GROUPED>
__global__ void __launch_bounds__(um::kThreads, 1)
    w8a8_umma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmX16, const __grid_constant__ CUtensorMap tmX32, Problem p) {
  using C = um::Cfg<MT>;
  constexpr int SR = C::RAW_STAGES, SO = C::OP_STAGES, XT = MT / 32, CH = C::CH;
  constexpr int kThreads = um::kThreads, kConv = um::kConvWarps * 32, kEpi = um::kEpiWarps * 32;
  constexpr int kEpiWarp0 = 2 + um::kConvWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = smem;
  uint8_t* xf = smem + SR * C::RAW;
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(xf + SO * C::XF);
  uint64_t* raw_empty = raw_full + SR;
  uint64_t* op_full = raw_empty + SR;
  uint64_t* op_empty = op_full + SO;
  uint64_t* acc_full = op_empty + SO;   // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint64_t* done_bar = acc_empty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ __align__(16) float s_sx[MT];
  __shared__ __align__(16) uint16_t s_ystage[16 * 128];  // epilogue staging: 16 tokens x 128 rows of bf16
  __shared__ int s_flag, s_issued, s_consumed;
  __shared__ int s_conv[2];         // k-blocks each converter group finished
  __shared__ volatile int s_abort;  // set after any timed-out wait: later waits are skipped
  __shared__ int tile_start_s[GROUPED ? 1025 : 1];
  __shared__ int rb[kMaxGrid + 1];
  __shared__ int wsum[kThreads / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // the barriers the first copies complete on come first; the rest after
    for (int i = 0; i < SR; ++i) mbar_init(&raw_full[i], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    // Thread 0 is the producer.  Dense problems issue their first weight
    // stages right here: they depend on nothing, and at decode sizes every
    // cycle before the first copy adds to the kernel time.
    if (!GROUPED) {
      // this CTA's stream-K range, as rb[] below tabulates it
      const int b0 = range_begin(p, blockIdx.x, gridDim.x);
      const int b1 = range_begin(p, blockIdx.x + 1, gridDim.x);
      const int pre = min(b1 - b0, p.pre_w > 0 && p.pre_w < SR ? p.pre_w : SR);
      const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      // one whole tile per CTA: no division
      int tile = p.per_cta == p.KB ? int(blockIdx.x) : b0 / p.KB, kb = b0 - tile * p.KB;
      TileCoord tc = decode_tile<MT, 128, GROUPED>(p, tile, nullptr);
      for (int r = 0; r < pre; ++r) {
        mbar_arrive_expect_tx(&raw_full[r], uint32_t(C::W_BYTES + um::x_box_rows<MT>(tc.rows) * kBK));
        tma_load_2d(raw + r * C::RAW, &tmW, &raw_full[r], kb * kBK, tc.w_row, pol_w);
        if (++kb == p.KB && r + 1 < pre) {
          kb = 0;
          tc = decode_tile<MT, 128, GROUPED>(p, ++tile, nullptr);
        }
      }
    }
    for (int i = 0; i < SR; ++i) mbar_init(&raw_empty[i], um::kConvWarps / 2);
    for (int i = 0; i < SO; ++i) {
      mbar_init(&op_full[i], um::kConvWarps / 2);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], um::kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_conv[0] = s_conv[1] = 0;
    s_abort = 0;
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmX16);
    tma_prefetch_desc(&tmX32);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, um::kTmemCols);
    tmem_relinquish();
  }

  int64_t I = p.total;
  if (GROUPED) {
    // per-expert tile counts from the device offsets (written by moe_sort)
    pdl_wait();
    const int NB = p.n_tiles;
    const int per = (p.E + kThreads - 1) / kThreads;
    int local = 0;
    for (int k = 0; k < per; ++k) {
      const int e = tid * per + k;
      if (e < p.E) {
        const int me = p.offsets[e + 1] - p.offsets[e];
        local += me > 0 ? NB * ((me + MT - 1) / MT) : 0;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int k = 0; k < per; ++k) {
      const int e = tid * per + k;
      if (e < p.E) {
        tile_start_s[e] = run;
        const int me = p.offsets[e + 1] - p.offsets[e];
        run += me > 0 ? NB * ((me + MT - 1) / MT) : 0;
      }
    }
    if (tid == kThreads - 1) tile_start_s[p.E] = run;
    __syncthreads();
    I = int64_t(tile_start_s[p.E]) * p.KB;
  }
  const int G = gridDim.x, b = blockIdx.x;
  for (int c = tid; c <= G; c += kThreads) rb[c] = GROUPED ? int(int64_t(c) * I / G) : range_begin(p, c, G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int begin = rb[b], end = rb[b + 1];
  const int KB = p.KB;
  const int n_it = end - begin;

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      const uint64_t pol_w = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int npre = n_it < SR ? n_it : SR;
      // weight stages issued at kernel entry; the other first-lap stages go
      // out right after the wait, into ring slots not yet used
      const int pre_w = (!GROUPED && p.pre_w > 0 && p.pre_w < npre) ? p.pre_w : npre;
      auto xrows = [&](int rows) { return um::x_box_rows<MT>(rows); };
      auto load_x = [&](int s_, int kb_, const TileCoord& t_) {
        const int xr = xrows(t_.rows);
        const CUtensorMap* m = xr == 16 ? &tmX16 : (xr == 32 ? &tmX32 : &tmX);
        tma_load_2d(raw + s_ * C::RAW + C::W_BYTES, m, &raw_full[s_], kb_ * kBK, t_.x_row, pol_x);
      };
      if (GROUPED) {  // weights do not depend on the previous kernel: issue them first (dense: done above)
        int tile = begin / KB, kb = begin - tile * KB;
        TileCoord tc = decode_tile<MT, 128, GROUPED>(p, tile, tile_start_s);
        for (int r = 0; r < npre; ++r) {
          mbar_arrive_expect_tx(&raw_full[r], uint32_t(C::W_BYTES + xrows(tc.rows) * kBK));
          tma_load_2d(raw + r * C::RAW, &tmW, &raw_full[r], kb * kBK, tc.w_row, pol_w);
          if (++kb == KB && r + 1 < npre) {
            kb = 0;
            tc = decode_tile<MT, 128, GROUPED>(p, ++tile, tile_start_s);
          }
        }
      }
      pdl_wait();
      int tile = begin / KB, kb = begin - tile * KB;
      TileCoord tc = decode_tile<MT, 128, GROUPED>(p, tile, tile_start_s);
      int issued = 0;
      for (int r = 0; r < n_it; ++r) {
        const int s = r % SR;
        if (r < pre_w) {
          load_x(s, kb, tc);
        } else {
          if (r >= npre && (s_abort || !mbar_wait(&raw_empty[s], uint32_t((r / SR - 1) & 1)))) {
            if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[s], uint32_t(C::W_BYTES + xrows(tc.rows) * kBK));
          tma_load_2d(raw + s * C::RAW, &tmW, &raw_full[s], kb * kBK, tc.w_row, pol_w);
          load_x(s, kb, tc);
        }
        ++issued;
        if (++kb == KB && r + 1 < n_it) {
          kb = 0;
          tc = decode_tile<MT, 128, GROUPED>(p, ++tile, tile_start_s);
        }
      }
      s_issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // The whole warp walks the k-blocks (waits and loop control warp-uniform)
    // and one elected lane issues: one thread issuing with a wait per block
    // cost ~0.3 us of issue overhead per block on GB300.
    constexpr uint32_t idesc = umma_idesc_f16_f32(128, MT);
    const uint32_t xf_base = smem_u32(xf);
    int kb = begin % KB, seg_kb0 = kb;
    int ch = -1;  // accumulator chunk (1024 K of one segment); region ch & 1
    int so = 0;
    uint32_t oph = 0;
    for (int r = 0; r < n_it; ++r) {
      const int kl = kb - seg_kb0;
      const bool chunk_start = (kl % kFlushBlocks) == 0;
      const bool seg_end = (kb == KB - 1) || (r == n_it - 1);
      const bool chunk_end = seg_end || (kl % kFlushBlocks) == kFlushBlocks - 1;
      if (chunk_start) ++ch;
      bool ok = true;
      if (chunk_start && ch >= 2) ok = mbar_wait_or_abort(&acc_empty[ch & 1], uint32_t(((ch >> 1) - 1) & 1), &s_abort);
      if (ok) ok = mbar_wait_or_abort(&op_full[so], oph, &s_abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (lane == 0) {
          if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + uint32_t((ch & 1) * CH * MT);
      const uint32_t a = tmem + uint32_t(C::ACC_COLS + so * 64);
      const uint64_t xd = umma_desc_k_sw128(xf_base + uint32_t(so * C::XF));
      if (elect_one()) {
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_f16_ts(d + uint32_t((s % CH) * MT), a + uint32_t(8 * s),
                      xd + uint64_t((((s >> 2) * (MT * kBK)) + (s & 3) * 32) >> 4), idesc,
                      (!chunk_start || s >= CH) ? 1u : 0u);
        umma_commit(&op_empty[so]);
        if (chunk_end) umma_commit(&acc_full[ch & 1]);
      }
      __syncwarp();
      if (seg_end) seg_kb0 = 0;
      if (++kb == KB) kb = 0;
      if (++so == SO) {
        so = 0;
        oph ^= 1u;
      }
    }
    // every MMA issued above has finished once this arrives
    if (elect_one()) umma_commit(done_bar);
    __syncwarp();
    const bool dok = mbar_wait(done_bar, 0);
    if (lane == 0 && !dok) atomicOr(p.err, DEVERR_TIMEOUT);
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------ converters
    pdl_wait();
    // Let the next kernel launch only once this one's inputs are final: a
    // dependent may prefetch weights before its own wait.
    pdl_launch_dependents();
    // Two groups of four warps take alternate k-blocks (two blocks in flight:
    // each warp's wait / load / convert / store / fence chain overlaps the
    // other group's); warp w of a group reaches tensor-memory lanes
    // 32*(w%4)..+31 and converts both 64-byte K halves of its rows.
    const int cw = warp - 2, q = warp & 3, grp = cw >> 2, gw = cw & 3;
    constexpr int kGrp = kConv / 2, XTG = 2 * XT;      // threads and activation tasks per group
    const int nl = 32 * q + lane;                       // weight row of the tile (tensor-memory lane)
    const uint32_t lane_off = uint32_t(32 * q) << 16;
    const uint32_t raw_base = smem_u32(raw), xf_base = smem_u32(xf);
    int consumed = 0, tile_cur = -1, rows_cur = 0;
    for (int r = grp; r < n_it; r += 2) {
      const int sr = r % SR, so = r % SO;
      const int tile = (begin + r) / KB;
      if (tile != tile_cur) {
        tile_cur = tile;
        rows_cur = decode_tile<MT, 128, GROUPED>(p, tile, tile_start_s).rows;
      }
      // one poll before the abort flag is read (a flag read per block measured
      // ~0.5 us over 16 blocks at M=64)
      const uint32_t pr = uint32_t((r / SR) & 1), po = uint32_t((r / SO - 1) & 1);
      bool ok = mbar_wait_try_first(&raw_full[sr], pr, &s_abort);
      if (ok && r >= SO) ok = mbar_wait_try_first(&op_empty[so], po, &s_abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t st = raw_base + uint32_t(sr * C::RAW);
      uint4 xv[XTG];
#pragma unroll
      for (int t = 0; t < XTG; ++t) {
        const int task = t * kGrp + gw * 32 + lane, xr = task >> 3, xc = task & 7;
        if (xr < rows_cur) xv[t] = lds128(st + uint32_t(C::W_BYTES + xr * kBK + ((xc ^ (xr & 7)) << 4)));
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = lds128(st + uint32_t(nl * kBK + (((4 * hh + c) ^ (nl & 7)) << 4)));
        uint32_t a[32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) i8x4_to_f16(word_of(v[c], i), a[8 * c + 2 * i], a[8 * c + 2 * i + 1]);
        tmem_st32(tmem + lane_off + uint32_t(C::ACC_COLS + so * 64 + 32 * hh), a);
      }
      const uint32_t xs = xf_base + uint32_t(so * C::XF);
#pragma unroll
      for (int t = 0; t < XTG; ++t) {
        const int task = t * kGrp + gw * 32 + lane, xr = task >> 3, xc = task & 7;
        if (xr < rows_cur) {
          uint32_t f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) i8x4_to_f16(word_of(xv[t], i), f[2 * i], f[2 * i + 1]);
          const uint32_t rowb = xs + uint32_t((xc >> 2) * (MT * kBK) + xr * kBK);
          const int j0 = 2 * (xc & 3);
          sts128(rowb + uint32_t((j0 ^ (xr & 7)) << 4), f[0], f[1], f[2], f[3]);
          sts128(rowb + uint32_t(((j0 + 1) ^ (xr & 7)) << 4), f[4], f[5], f[6], f[7]);
        }
      }
      tmem_wait_st();
      // the raw stage was read and the f16 operand written through the
      // generic proxy; TMA (next raw fill) and the tensor cores read or write
      // through the async proxy
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[sr]);
        mbar_arrive(&op_full[so]);
      }
      ++consumed;
    }
    if (gw == 0 && lane == 0) s_conv[grp] = consumed;
  } else {
    // ------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int nl = 32 * q + lane;                       // weight row of the tile (tensor-memory lane)
    const int etid = tid - kEpiWarp0 * 32;
    const uint32_t trow = tmem + (uint32_t(32 * q) << 16);
    const uint32_t tsum = trow + uint32_t(C::ISUM_COL);
    int tile = begin / KB, kb = begin - tile * KB;
    int seg_kb0 = kb;
    bool first_seg = true;
    int ch = -1;
    for (int r = 0; r < n_it; ++r) {
      const int kl = kb - seg_kb0;
      const bool seg_end = (kb == KB - 1) || (r == n_it - 1);
      const bool chunk_end = seg_end || (kl % kFlushBlocks) == kFlushBlocks - 1;
      if ((kl % kFlushBlocks) == 0) ++ch;
      if (chunk_end) {
        // add region ch & 1, rounded to int32 (exact), into the segment's sums
        // and hand the region back to the tensor cores
        bool ok = !s_abort && mbar_wait(&acc_full[ch & 1], uint32_t((ch >> 1) & 1));
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        } else {
          tc_fence_after();
          const bool first_chunk = kl < kFlushBlocks;
          // DW columns per round trip: every load of a piece is issued before one wait
          constexpr int DW = (CH + 1) * 32 <= 96 ? 32 : 16;
#pragma unroll
          for (int h = 0; h < MT / DW; ++h) {
            uint32_t sm[DW], f[CH][DW];
            if constexpr (DW == 32) {
              if (!first_chunk) tmem_ld32(tsum + uint32_t(DW * h), sm);
#pragma unroll
              for (int c = 0; c < CH; ++c) tmem_ld32(trow + uint32_t(((ch & 1) * CH + c) * MT + DW * h), f[c]);
            } else {
              if (!first_chunk) tmem_ld16(tsum + uint32_t(DW * h), sm);
#pragma unroll
              for (int c = 0; c < CH; ++c) tmem_ld16(trow + uint32_t(((ch & 1) * CH + c) * MT + DW * h), f[c]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < DW; ++j) {
              int32_t v = first_chunk ? 0 : int32_t(sm[j]);
#pragma unroll
              for (int c = 0; c < CH; ++c) v += __float2int_rn(__uint_as_float(f[c][j]));
              sm[j] = uint32_t(v);
            }
            if constexpr (DW == 32) tmem_st32(tsum + uint32_t(DW * h), sm); else tmem_st16(tsum + uint32_t(DW * h), sm);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[ch & 1]);
        }
      }
      if (seg_end) {
        // ---- segment end: tile `tile`, k-blocks [seg_kb0, kb]
        const TileCoord tc = decode_tile<MT, 128, GROUPED>(p, tile, tile_start_s);
        const bool whole = (seg_kb0 == 0) && (kb == KB - 1);
        bool do_epi = whole;
        if (!whole) {
          int32_t* my = p.slots + (2 * b + (first_seg ? 0 : 1)) * int64_t(C::SLOT) + nl;
#pragma unroll
          for (int h = 0; h < MT / 16; ++h) {
            uint32_t sm[16];
            tmem_ld16(tsum + uint32_t(16 * h), sm);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) my[(16 * h + j) * 128] = int32_t(sm[j]);
          }
          named_bar_sync(1, kEpi);
          if (etid == 0) {
            const uint32_t nb = uint32_t(kb - seg_kb0 + 1);
            const uint32_t old = atom_add_acq_rel_gpu(&p.counters[tile], nb);
            const int last = (old + nb == uint32_t(KB)) ? 1 : 0;
            if (last) p.counters[tile] = 0;  // every contributor has arrived; ready for the next call
            s_flag = last;
          }
          named_bar_sync(1, kEpi);
          do_epi = s_flag != 0;
        }
        if (do_epi) {
          // do_epi is uniform over the epilogue warps (whole, or s_flag)
          if (etid < MT) s_sx[etid] = etid < tc.rows ? __ldg(p.sx + tc.x_row + etid) : 0.f;
          named_bar_sync(1, kEpi);
          const int c0 = whole ? 0 : cta_of(rb, G, tile * KB), c1 = whole ? -1 : cta_of(rb, G, tile * KB + KB - 1);
          const int n = tc.n0 + nl;
          const float swv = n < p.N ? __ldg(p.sw + tc.sw_base + n) : 0.f;  // rows past N are never stored
          // add the other contributors' partial sums into the tensor-memory
          // sums: all MT values of a contributor are loaded in one batch
          for (int cc = c0; cc <= c1; ++cc) {
            // skip self and CTAs with an empty range (more CTAs than iterations)
            if (cc == b || rb[cc + 1] == rb[cc]) continue;
            const int first_tile = rb[cc] / KB;
            const int32_t* sl = p.slots + (2 * int64_t(cc) + (first_tile == tile ? 0 : 1)) * int64_t(C::SLOT) + nl;
            int32_t v[MT];
#pragma unroll
            for (int j = 0; j < MT; ++j) v[j] = __ldcg(sl + j * 128);
#pragma unroll
            for (int h = 0; h < MT / 16; ++h) {
              uint32_t sm[16];
              tmem_ld16(tsum + uint32_t(16 * h), sm);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) sm[j] = uint32_t(int32_t(sm[j]) + v[16 * h + j]);
              tmem_st16(tsum + uint32_t(16 * h), sm);
            }
            tmem_wait_st();
          }
#pragma unroll
          for (int h = 0; h < MT / 16; ++h) {
            uint32_t sm[16];
            tmem_ld16(tsum + uint32_t(16 * h), sm);
            tmem_wait_ld();
            int32_t acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = int32_t(sm[j]);
            // dequantize 16 tokens of this row into the staging tile
            // [16 tokens][128 rows], then write whole 16-byte pieces of y rows
            float sxv[16];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 t = *reinterpret_cast<const float4*>(&s_sx[16 * h + j]);
              sxv[j] = t.x;
              sxv[j + 1] = t.y;
              sxv[j + 2] = t.z;
              sxv[j + 3] = t.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              s_ystage[j * 128 + nl] = f32_to_bf16_bits(__fmul_rn(__fmul_rn(__int2float_rn(acc[j]), sxv[j]), swv));
            named_bar_sync(1, kEpi);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int piece = i * kEpi + etid, j = piece >> 4, c8 = piece & 15;  // 16 pieces of 8 per token
              const int m = 16 * h + j, nn = tc.n0 + 8 * c8;
              if (m < tc.rows && nn < p.N) {
                const uint4 v = *reinterpret_cast<const uint4*>(&s_ystage[j * 128 + 8 * c8]);
                st_global_v4(p.y + int64_t(tc.x_row + m) * p.N + nn, v);
              }
            }
            named_bar_sync(1, kEpi);
          }
          named_bar_sync(1, kEpi);  // s_sx is rewritten by the next segment
        }
        tc_fence_before();
        first_seg = false;
        seg_kb0 = 0;
      }
      if (++kb == KB) {
        kb = 0;
        ++tile;
      }
    }
  }
  __syncthreads();
  // Drain: on the normal path every issued stage was consumed.  After a
  // timeout, wait (bounded) for copies still in flight before exiting.
  if (tid == 0) {
    // blocks 0 .. 2*c0-2 went to group 0, 1 .. 2*c1-1 to group 1: the contiguous prefix converted
    const int done = min(2 * s_conv[0], 2 * s_conv[1] + 1);
    for (int r = done; r < s_issued; ++r) mbar_wait(&raw_full[r % SR], uint32_t((r / SR) & 1));
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, um::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
static constexpr int pick_mt(int64_t M) { return M <= 8 ? 8 : (M <= 16 ? 16 : (M <= 32 ? 32 : 64)); }

static constexpr size_t slots_bytes(int sms, int mt) { return size_t(2) * sms * kBN * mt * 4; }
// Token tile the partial-sum slots are sized for: the tcgen05 kernel runs
// tiles of at least 32 tokens (a forced schedule may run it for any M).
static constexpr int slots_mt(int64_t M) { return pick_mt(M) < 32 ? 32 : pick_mt(M); }

// Workspace layout: [counters: kCounterBytes][xq, sx: fused call only][partial-sum slots]
size_t ws_w8a8_linear(int64_t M, int64_t K, int64_t N) {
  DevInfo d;
  if (device_info(&d) != FQ_OK || M < 0 || K < 0 || N < 0) return 0;
  return kCounterBytes + slots_bytes(d.sm_count, slots_mt(M));
}

size_t ws_w8a8_quant_linear(int64_t M, int64_t K, int64_t N) {
  const size_t g = ws_w8a8_linear(M, K, N);
  if (!g) return 0;
  return align_up(size_t(M) * size_t(K), 256) + align_up(size_t(M) * 4, 256) + g;
}

size_t ws_w8a8_grouped_linear(int64_t R, int64_t K, int64_t N, int64_t E) {
  DevInfo d;
  if (device_info(&d) != FQ_OK || R < 0 || K < 0 || N < 0 || E < 0) return 0;
  return kCounterBytes + slots_bytes(d.sm_count, 64);
}

template <int MT, int CW, bool GROUPED, bool FQ = false>
static cudaError_t launch_gemm(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid,
                               cudaStream_t s, bool pdl) {
  using C = Cfg<MT, CW, FQ>;
  auto k = w8a8_gemm_kernel<MT, CW, GROUPED, FQ>;
  static uint64_t attr_done = 0;  // one bit per device id
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch(k, dim3(grid), dim3(C::THREADS), size_t(C::SMEM), s, pdl, *tw, *tx, p);
}

template <int MT, bool GROUPED>
static cudaError_t launch_umma_gemm(const CUtensorMap* tw, const CUtensorMap* tx, const CUtensorMap* tx16,
                                    const CUtensorMap* tx32, const Problem& p, int grid, cudaStream_t s, bool pdl) {
  using C = um::Cfg<MT>;
  auto k = w8a8_umma_kernel<MT, GROUPED>;
  static uint64_t attr_done = 0;  // one bit per device id
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch(k, dim3(grid), dim3(um::kThreads), size_t(C::SMEM), s, pdl, *tw, *tx, *tx16, *tx32, p);
}

template <int MT>
static cudaError_t launch_cluster_gemm(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid,
                                       cudaStream_t s, bool pdl) {
  using C = CCfg<MT, 2, 4, 4>;
  auto k = w8a8_cluster_kernel<MT, 2, 4, 4>;
  static uint64_t attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch_cluster(k, dim3(grid), dim3(C::THREADS), size_t(C::SMEM), s, pdl, 4u, *tw, *tx, p);
}

// Schedule override for tests and cliff studies: FQ_FORCE_SCHEDULE = dp |
// cluster | streamk | umma (read on every call).  A forced choice the shape
// cannot take is ignored.  FQ_DEBUG_SCHEDULE=1 prints each decision to stderr.
enum Sched { SCHED_AUTO = 0, SCHED_DP = 1, SCHED_CLUSTER = 2, SCHED_STREAMK = 3, SCHED_UMMA = 4 };
static int forced_schedule() {
  const char* v = std::getenv("FQ_FORCE_SCHEDULE");
  if (!v) return SCHED_AUTO;
  if (!std::strcmp(v, "dp")) return SCHED_DP;
  if (!std::strcmp(v, "cluster")) return SCHED_CLUSTER;
  if (!std::strcmp(v, "streamk")) return SCHED_STREAMK;
  if (!std::strcmp(v, "umma")) return SCHED_UMMA;
  return SCHED_AUTO;
}
// Stages the producer keeps in flight.  Every CTA asking for its whole ring
// at once (~200 KB per SM) makes HBM interleave all of them, so the first
// stage lands only when most of the data has (~3.6 us) and the consumers
// start late; with ~120 KB per SM in flight the bandwidth holds and the first
// stages land sooner.  Measured on the 224-row tiles (K=1024, N=32768):
// 4 stages 8.3-8.7 us at M <= 8 against 9.3-9.8 for the whole ring (7), 3
// stages 8.4-9.0, 2 stages 9.6-9.8.  FQ_STAGES_AHEAD overrides (studies).
static int stages_ahead(int stage_bytes) {
  if (const char* v = std::getenv("FQ_STAGES_AHEAD")) return std::atoi(v);
  const int n = (122880 + stage_bytes / 2) / stage_bytes;
  return n < 2 ? 2 : n;
}
static void debug_schedule(const char* op, int64_t M, int64_t K, int64_t N, int mt, const char* sched, int grid) {
  const char* v = std::getenv("FQ_DEBUG_SCHEDULE");
  if (v && v[0] == '1')
    std::fprintf(stderr, "fq: %s M=%lld K=%lld N=%lld mt=%d schedule=%s grid=%d\n", op, (long long)M, (long long)K,
                 (long long)N, mt, sched, grid);
}

// Shared by the dense and fused entry points.  `counters` is the fixed
// counter block at the head of the workspace; `slots` the partial-sum area.
// The fused op runs as one launch when the dense schedule would stream one
// whole 224-row tile per CTA and the whole quantized activation tile fits in
// shared memory: each CTA quantizes the activations itself after the previous
// kernel has finished.  That beats a separate quant launch while every row
// has a consumer warp of its own (K=1024, N=32768 on GB300: M=9 10.8 -> 10.4
// us); with 15 or 16 rows two warps quantize two rows one after the other
// (M=16: 11.4 against 10.7 us with two launches).
static bool quant_in_gemm(int64_t M, int64_t K, int64_t N, const DevInfo& d) {
  const int mt = pick_mt(M);
  if (mt > 16 || M > mt || K > kFuseKMax) return false;
  if (M > 14) return false;  // one row per consumer warp of the 224-row kernel
  const int force = forced_schedule();
  const int64_t tiles224 = (N + 223) / 224;
  if (force == SCHED_DP) return tiles224 <= kMaxGrid;
  if (force != SCHED_AUTO) return false;
  return tiles224 <= d.sm_count && tiles224 * 4 >= int64_t(d.sm_count) * 3;
}

// Weight stages a dense GEMM issues before its wait on the previous kernel.
// Copies issued early sit ahead of everything the kernel requests after the
// wait, so the right number depends on what comes then.  Measured on GB300
// (K=1024, N=32768, chained calls): the 224-row kernel takes three of its
// four in-flight stages when the previous kernel is another GEMM (M <= 8
// 7.85 -> 7.75 us, M = 16 9.1 -> 9.0; one or two stages are slower), but
// behind the per-token quant - its own, in the one-launch fused op, or the
// fused op's separate quant launch - one stage: M <= 8 fused 8.7-9.4 ->
// 7.9-8.7 us, M = 16 fused 11.2 -> 10.7.  The tcgen05 kernel takes three
// of its eight raw stages either way: M = 32 10.6 -> 10.1 us, M = 64 11.9 ->
// 11.7, fused 12.4 -> 11.9 and 14.0 -> 13.7.  The small linear's cluster
// kernel keeps all of its stages (fewer measured slower at M <= 16).
constexpr int kPreWaitAfterGemm = 3;
constexpr int kPreWaitAfterQuant = 1;
constexpr int kPreWaitUmma = 3;

fq_status run_w8a8_dense(const int8_t* xq, const float* sx, int64_t M, int64_t K, const int8_t* w_nk, const float* sw,
                         int64_t N, uint16_t* y, uint32_t* counters, void* slots, size_t slots_avail, cudaStream_t s,
                         const DevInfo& d, bool after_quant) {
  const int mt = pick_mt(M);
  const int64_t m_tiles = (M + mt - 1) / mt;
  const int KB = int((K + kBK - 1) / kBK);
  // Schedule.  When tiles of 224 weight rows (14 consumer warps) give between
  // 3/4 of and one tile per SM, every CTA streams one whole tile: no split-K,
  // no partial sums - for token tiles up to 16; at 32 the tcgen05 kernel is
  // ahead (K=1024, N=32768 on GB300: 10.8 against 11.4 us).  Otherwise
  // 128-row tiles are split stream-K over one CTA per SM.
  const int64_t tiles224 = ((N + 223) / 224) * m_tiles;
  bool data_parallel = mt <= 16 && tiles224 <= d.sm_count && tiles224 * 4 >= int64_t(d.sm_count) * 3;
  // Few tiles (small N): 32-row tiles, each split over K by a cluster of 4 CTAs
  // with a distributed-shared-memory reduction, when that fills >= 1/2 the GPU
  // (every token tile: with its k-split warps it beats the tcgen05 kernel at 64).
  const int64_t ctas_cl = ((N + 31) / 32) * m_tiles * 4;
  bool cluster = !data_parallel && ctas_cl <= d.sm_count && ctas_cl * 2 >= d.sm_count && KB >= 4;
  const int force = forced_schedule();
  if (force == SCHED_DP && mt <= 32 && tiles224 <= kMaxGrid) {
    data_parallel = true;
    cluster = false;
  } else if (force == SCHED_CLUSTER && KB >= 4 && ctas_cl <= (int64_t(1) << 30)) {
    data_parallel = false;
    cluster = true;
  } else if (force == SCHED_STREAMK || force == SCHED_UMMA) {
    data_parallel = cluster = false;
  }
  // Stream-K with token tiles of 32 or 64 runs on the tcgen05 kernel (the
  // mma.sync kernel is instruction-bound there).
  const bool umma = !data_parallel && !cluster &&
                    (force == SCHED_UMMA ? true : (force == SCHED_STREAMK ? false : mt >= 32));
  const int mt_run = umma && mt < 32 ? 32 : mt;
  if (cluster) {
    Problem p = {};
    p.M = int(M);
    p.N = int(N);
    p.K = int(K);
    p.KB = KB;
    p.m_tiles = int(m_tiles);
    p.n_tiles = int((N + 31) / 32);
    p.total = 0;
    p.sx = sx;
    p.sw = sw;
    p.y = y;
    p.err = d.err_word;
    p.w_reuse = m_tiles > 1 ? 1 : 0;
    CUtensorMap tw_map, tx_map;
    if (!tensor_map_u8_2d(&tw_map, w_nk, uint64_t(K), uint64_t(N), uint64_t(K), kBK, 32u) ||
        !tensor_map_u8_2d(&tx_map, xq, uint64_t(K), uint64_t(M), uint64_t(K), kBK, uint32_t(mt)))
      return FQ_ERR_CUDA;
    const CUtensorMap* tw = &tw_map;
    const CUtensorMap* tx = &tx_map;
    const int grid = int(ctas_cl);
    debug_schedule("w8a8_linear", M, K, N, mt, "cluster4", grid);
    const bool pdl = pdl_enabled();
    cudaError_t e;
    switch (mt) {
      case 8: e = launch_cluster_gemm<8>(tw, tx, p, grid, s, pdl); break;
      case 16: e = launch_cluster_gemm<16>(tw, tx, p, grid, s, pdl); break;
      case 32: e = launch_cluster_gemm<32>(tw, tx, p, grid, s, pdl); break;
      default: e = launch_cluster_gemm<64>(tw, tx, p, grid, s, pdl); break;
    }
    return cuda_status(e);
  }
  const int64_t n_tiles = data_parallel ? (N + 223) / 224 : (N + kBN - 1) / kBN;
  const int64_t m_tiles_run = (M + mt_run - 1) / mt_run;
  const int64_t tiles = m_tiles_run * n_tiles;
  if (tiles > kMaxTiles || int64_t(tiles) * KB > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  if (!data_parallel && slots_avail < slots_bytes(d.sm_count, mt_run)) return FQ_ERR_WORKSPACE;
  Problem p = {};
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.KB = KB;
  p.m_tiles = int(m_tiles_run);
  p.n_tiles = int(n_tiles);
  p.total = tiles * KB;
  p.sx = sx;
  p.sw = sw;
  p.y = y;
  p.counters = counters;
  p.slots = static_cast<int32_t*>(slots);
  p.err = d.err_word;
  p.w_reuse = m_tiles_run > 1 ? 1 : 0;
  p.ahead = stages_ahead(int((data_parallel ? 224 : kBN) * kBK + mt_run * kBK));
  const uint32_t bn = data_parallel ? 224u : uint32_t(kBN);
  CUtensorMap tw_map, tx_map;
  if (!tensor_map_u8_2d(&tw_map, w_nk, uint64_t(K), uint64_t(N), uint64_t(K), kBK, bn) ||
      !tensor_map_u8_2d(&tx_map, xq, uint64_t(K), uint64_t(M), uint64_t(K), kBK, uint32_t(mt_run)))
    return FQ_ERR_CUDA;
  const CUtensorMap* tw = &tw_map;
  const CUtensorMap* tx = &tx_map;
  // tcgen05 path: at least 4 k-blocks per CTA (its fixed cost - tensor-memory
  // set-up, pipeline fill, epilogue - and a tile's hand-off grow with the CTAs
  // sharing the tile)
  const int64_t work = umma ? (p.total + 3) / 4 : p.total;
  int grid = data_parallel ? int(tiles) : int(work < d.sm_count ? (work > 0 ? work : 1) : d.sm_count);
  if (umma) {
    const int g = whole_tile_grid(tiles, d.sm_count);
    if (g > 0 && g <= grid) grid = g;
  }
  p.per_cta = p.total % grid == 0 ? int(p.total / grid) : 0;
  // (measured on the whole-tile schedules; the stream-K mma.sync form keeps its default)
  p.pre_w = umma ? kPreWaitUmma : (data_parallel ? (after_quant ? kPreWaitAfterQuant : kPreWaitAfterGemm) : 0);
  debug_schedule("w8a8_linear", M, K, N, mt_run, data_parallel ? "dp224" : (umma ? "umma" : "streamk"), grid);
  const bool pdl = pdl_enabled();
  cudaError_t e;
  if (umma) {
    CUtensorMap tx16, tx32;  // smaller activation boxes for tiles with few token rows
    if (!tensor_map_u8_2d(&tx16, xq, uint64_t(K), uint64_t(M), uint64_t(K), kBK, 16u) ||
        !tensor_map_u8_2d(&tx32, xq, uint64_t(K), uint64_t(M), uint64_t(K), kBK, 32u))
      return FQ_ERR_CUDA;
    e = mt_run == 32 ? launch_umma_gemm<32, false>(tw, tx, &tx16, &tx32, p, grid, s, pdl)
                     : launch_umma_gemm<64, false>(tw, tx, &tx16, &tx32, p, grid, s, pdl);
  } else if (data_parallel) {
    e = mt == 8    ? launch_gemm<8, 14, false>(tw, tx, p, grid, s, pdl)
        : mt == 16 ? launch_gemm<16, 14, false>(tw, tx, p, grid, s, pdl)
                   : launch_gemm<32, 14, false>(tw, tx, p, grid, s, pdl);
  } else {
    switch (mt) {
      case 8: e = launch_gemm<8, 8, false>(tw, tx, p, grid, s, pdl); break;
      case 16: e = launch_gemm<16, 8, false>(tw, tx, p, grid, s, pdl); break;
      case 32: e = launch_gemm<32, 8, false>(tw, tx, p, grid, s, pdl); break;
      default: e = launch_gemm<64, 8, false>(tw, tx, p, grid, s, pdl); break;
    }
  }
  return cuda_status(e);
}

}  // namespace fq

using namespace fq;

static fq_status check_linear_args(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K < 0 || N < 0 || K % 16 || N % 16) return FQ_ERR_SHAPE;
  if (K > 131072 || N > (int64_t(1) << 24) || M > (int64_t(1) << 24)) return FQ_ERR_SHAPE;
  return FQ_OK;
}

extern "C" __attribute__((visibility("default"))) fq_status w8a8_linear(const int8_t* xq, const float* sx, int64_t M, int64_t K, const int8_t* w_nk,
                                 const float* sw, int64_t N, uint16_t* y, void* ws, size_t ws_bytes,
                                 fq_stream_t stream) {
  fq_status st = check_linear_args(M, K, N);
  if (st != FQ_OK) return st;
  if (M == 0 || N == 0) return FQ_OK;
  if (!xq || !sx || !w_nk || !sw || !y) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(sx) || !aligned16(w_nk) || !aligned16(sw) || !aligned16(y)) return FQ_ERR_ALIGN;
  DevInfo d;
  if ((st = device_info(&d)) != FQ_OK) return st;
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(y, 0, size_t(M) * size_t(N) * 2, reinterpret_cast<cudaStream_t>(stream));
    return cuda_status(e);
  }
  if (!ws || ws_bytes < kCounterBytes) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  return run_w8a8_dense(xq, sx, M, K, w_nk, sw, N, y, reinterpret_cast<uint32_t*>(w8), w8 + kCounterBytes,
                        ws_bytes - kCounterBytes, reinterpret_cast<cudaStream_t>(stream), d, false);
}

extern "C" __attribute__((visibility("default"))) fq_status w8a8_quant_linear(const uint16_t* x, int64_t M, int64_t K, const int8_t* w_nk, const float* sw,
                                       int64_t N, uint16_t* y, int8_t* xq_out, float* sx_out, void* ws,
                                       size_t ws_bytes, fq_stream_t stream) {
  fq_status st = check_linear_args(M, K, N);
  if (st != FQ_OK) return st;
  if (M == 0) return FQ_OK;
  if (!x || !w_nk || !sw || !y) return FQ_ERR_NULL;
  if (!aligned16(x) || !aligned16(w_nk) || !aligned16(sw) || !aligned16(y) || (xq_out && !aligned16(xq_out)) ||
      (sx_out && !aligned16(sx_out)))
    return FQ_ERR_ALIGN;
  DevInfo d;
  if ((st = device_info(&d)) != FQ_OK) return st;
  const size_t xq_b = align_up(size_t(M) * size_t(K), 256), sx_b = align_up(size_t(M) * 4, 256);
  if (!ws || ws_bytes < kCounterBytes + xq_b + sx_b) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  int8_t* xq = xq_out ? xq_out : reinterpret_cast<int8_t*>(w8 + kCounterBytes);
  float* sx = sx_out ? sx_out : reinterpret_cast<float*>(w8 + kCounterBytes + xq_b);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // validate the GEMM part before launching the quant
  if (N > 0 && K > 0 && ws_bytes - kCounterBytes - xq_b - sx_b < slots_bytes(d.sm_count, slots_mt(M)))
    return FQ_ERR_WORKSPACE;
  if (N > 0 && K > 0 && quant_in_gemm(M, K, N, d)) {
    // one launch: every CTA quantizes the (small) activation tile itself
    const int mt = pick_mt(M);
    const int64_t tiles = (N + 223) / 224;
    Problem p = {};
    p.M = int(M);
    p.N = int(N);
    p.K = int(K);
    p.KB = int((K + kBK - 1) / kBK);
    p.m_tiles = 1;
    p.n_tiles = int(tiles);
    p.total = tiles * p.KB;
    p.per_cta = p.KB;  // one whole tile per CTA
    p.pre_w = kPreWaitAfterQuant;  // the CTA's own quant comes right after the wait
    p.sw = sw;
    p.y = y;
    p.counters = reinterpret_cast<uint32_t*>(w8);
    p.err = d.err_word;
    p.x16 = x;
    p.xq_out = xq_out;
    p.sx_out = sx_out;
    p.ahead = stages_ahead(224 * kBK);
    // With 3 to 8 rows the CTA's own quant holds its consumers back for a
    // while after the wait; one more stage in flight keeps the weight stream
    // going meanwhile (GB300, K=1024, N=32768: M = 3 / 4 / 7 / 8 8.1 / 8.3 /
    // 8.35 / 8.7 -> 7.7 / 7.75 / 7.8 / 8.2 us; with 1 or 2 rows, or 16-token
    // tiles, the window of the plain GEMM measured as fast or faster).
    if (mt == 8 && M >= 3 && !std::getenv("FQ_STAGES_AHEAD")) p.ahead += 1;
    CUtensorMap tw_map;
    if (!tensor_map_u8_2d(&tw_map, w_nk, uint64_t(K), uint64_t(N), uint64_t(K), kBK, 224u)) return FQ_ERR_CUDA;
    debug_schedule("w8a8_quant_linear", M, K, N, mt, "dp224+quant", int(tiles));
    const bool pdl = pdl_enabled();
    return cuda_status(mt == 8 ? launch_gemm<8, 14, false, true>(&tw_map, &tw_map, p, int(tiles), s, pdl)
                               : launch_gemm<16, 14, false, true>(&tw_map, &tw_map, p, int(tiles), s, pdl));
  }
  // the quant's output is this call's activations: the GEMM may launch early
  if ((st = quant_int8_launch(x, M, K, xq, sx, stream, true)) != FQ_OK) return st;
  if (N == 0) return FQ_OK;
  if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, size_t(M) * size_t(N) * 2, s));
  return run_w8a8_dense(xq, sx, M, K, w_nk, sw, N, y, reinterpret_cast<uint32_t*>(w8),
                        w8 + kCounterBytes + xq_b + sx_b, ws_bytes - kCounterBytes - xq_b - sx_b, s, d, true);
}

extern "C" __attribute__((visibility("default"))) fq_status w8a8_grouped_linear(const int8_t* xq, const float* sx, const int32_t* offsets, int64_t R,
                                         int64_t E, int64_t K, const int8_t* w_enk, const float* sw_en, int64_t N,
                                         uint16_t* y, void* ws, size_t ws_bytes, fq_stream_t stream) {
  fq_status st = check_linear_args(R, K, N);
  if (st != FQ_OK) return st;
  if (E <= 0 || E > 1024 || E * N > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  if (R == 0 || N == 0) return FQ_OK;
  if (K == 0) return FQ_ERR_SHAPE;
  if (!xq || !sx || !offsets || !w_enk || !sw_en || !y) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(sx) || !aligned16(offsets) || !aligned16(w_enk) || !aligned16(sw_en) ||
      !aligned16(y))
    return FQ_ERR_ALIGN;
  DevInfo d;
  if ((st = device_info(&d)) != FQ_OK) return st;
  constexpr int mt = 64;
  const int64_t n_tiles = (N + kBN - 1) / kBN;
  const int64_t max_tiles = n_tiles * ((R + mt - 1) / mt + E);
  if (max_tiles > kMaxTiles) return FQ_ERR_SHAPE;
  const size_t need = kCounterBytes + slots_bytes(d.sm_count, mt);
  if (!ws || ws_bytes < need) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  Problem p = {};
  p.M = int(R);
  p.N = int(N);
  p.K = int(K);
  p.KB = int((K + kBK - 1) / kBK);
  p.n_tiles = int(n_tiles);
  p.m_tiles = 0;
  p.total = 0;
  p.sx = sx;
  p.sw = sw_en;
  p.y = y;
  p.counters = static_cast<uint32_t*>(ws);
  p.slots = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.err = d.err_word;
  p.offsets = offsets;
  p.E = int(E);
  p.w_reuse = 1;
  CUtensorMap tw_map, tx_map;
  if (!tensor_map_u8_2d(&tw_map, w_enk, uint64_t(K), uint64_t(E * N), uint64_t(K), kBK, kBN) ||
      !tensor_map_u8_2d(&tx_map, xq, uint64_t(K), uint64_t(R), uint64_t(K), kBK, uint32_t(mt)))
    return FQ_ERR_CUDA;
  const CUtensorMap* tw = &tw_map;
  const CUtensorMap* tx = &tx_map;
  const bool umma = forced_schedule() != SCHED_STREAMK;
  debug_schedule("w8a8_grouped_linear", R, K, N, mt, umma ? "umma" : "streamk", d.sm_count);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tx16, tx32;
  if (umma && (!tensor_map_u8_2d(&tx16, xq, uint64_t(K), uint64_t(R), uint64_t(K), kBK, 16u) ||
               !tensor_map_u8_2d(&tx32, xq, uint64_t(K), uint64_t(R), uint64_t(K), kBK, 32u)))
    return FQ_ERR_CUDA;
  return cuda_status(umma ? launch_umma_gemm<mt, true>(tw, tx, &tx16, &tx32, p, d.sm_count, s, pdl_enabled())
                          : launch_gemm<mt, 8, true>(tw, tx, p, d.sm_count, s, pdl_enabled()));
}

// ================================================================ no-allocation variant
//
// w8a8_linear_noalloc: the same W8A8 linear for callers that cannot allocate
// device memory - code running where cudaMalloc is unavailable or forbidden
// (inside an allocator-free runtime, a plugin that must not touch the
// caller's memory pool, or code that owns no device memory at all).  Its
// split-K scratch is a fixed file-scope device array instead of a caller
// workspace.
namespace fq {
namespace noalloc {
constexpr int64_t kMaxM = 64;                                    // one token tile of 64
constexpr int64_t kMaxTilesNA = 4096;                            // N <= 4096 * 128 = 524288
constexpr int kMaxCtas = 160;                                    // one CTA per SM; GB300 has 152
constexpr size_t kCountersNA = size_t(kMaxTilesNA) * 4;         // 16 KiB of arrival counters
constexpr size_t kSlotsNA = size_t(2) * kMaxCtas * kBN * 64 * 4;  // 10 MiB of int32 partial sums
constexpr size_t kScratchBytes = kCountersNA + kSlotsNA;
// the partial sums of every schedule a call within the limits can take (token
// tiles up to 64, one CTA per SM), and one arrival counter per 128-row tile
static_assert(kSlotsNA >= slots_bytes(kMaxCtas, slots_mt(kMaxM)), "partial-sum area too small");
static_assert(size_t(kMaxTilesNA) * 4 <= kCountersNA, "counter area too small");
static_assert(slots_mt(kMaxM) == kMaxM, "M <= kMaxM is one token tile on every schedule");
}  // namespace noalloc

// Held by every device that loads this library, for the life of the process.
static __device__ __align__(256) uint8_t g_w8a8_noalloc_scratch[noalloc::kScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64] = {};

// Device address of the scratch array on the current device (set-up once per
// device, with that device current).  The host-side name of the array is only
// a stand-in for the symbol and must never be passed to a kernel.
static fq_status noalloc_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (dev < 0 || dev >= 64) return FQ_ERR_UNSUPPORTED_DEVICE;
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_w8a8_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FQ_OK;
}
}  // namespace fq

extern "C" __attribute__((visibility("default"))) fq_status w8a8_linear_noalloc(
    const int8_t* xq, const float* sx, int64_t M, int64_t K, const int8_t* w_nk, const float* sw, int64_t N,
    uint16_t* y, fq_stream_t stream) {
  fq_status st = check_linear_args(M, K, N);
  if (st != FQ_OK) return st;
  if (M > noalloc::kMaxM) return FQ_ERR_SHAPE;
  if (((N + kBN - 1) / kBN) > noalloc::kMaxTilesNA) return FQ_ERR_SHAPE;
  if (M == 0 || N == 0) return FQ_OK;
  if (!xq || !sx || !w_nk || !sw || !y) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(sx) || !aligned16(w_nk) || !aligned16(sw) || !aligned16(y)) return FQ_ERR_ALIGN;
  DevInfo d;
  if ((st = device_info(&d)) != FQ_OK) return st;
  if (d.sm_count > noalloc::kMaxCtas) return FQ_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, size_t(M) * size_t(N) * 2, s));
  void* scratch = nullptr;
  if ((st = noalloc_scratch(d.id, &scratch)) != FQ_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  const int64_t tiles = (N + kBN - 1) / kBN;  // M <= 64: one token tile
  // The array keeps the previous call's contents: the arrival counters this
  // call uses must start at zero.
  cudaError_t e = cudaMemsetAsync(base, 0, size_t(tiles) * 4, s);
  if (e != cudaSuccess) return cuda_status(e);
  return run_w8a8_dense(xq, sx, M, K, w_nk, sw, N, y, reinterpret_cast<uint32_t*>(base), base + noalloc::kCountersNA,
                        noalloc::kSlotsNA, s, d, false);
}
