// Block-scaled FP8 grouped einsum, the consumer of the packed UE8M0
// activation scales ("SGLang PR #34277 digest": motivation and
// implementation breakdown item 3 - deep_gemm.fp8_einsum reads the
// TMA-aligned packed scales; packed and fp32 scales must give bit-identical
// outputs).
//
//   Y[t, g, n] = bf16( sum_kb sx[t,g,kb] * sw[g,kb,n/128] * sum_{d in kb} xq[t,g,d] * W[g,d,n] )
//
// GB300 design:
//  * Swap-AB tiles of 128 weight rows (n) x MT tokens, one per (g, n-block,
//    token tile); weights E4M3 [G, N, D] K-major, activations E4M3 [T, G, D].
//  * Engine: warp-level e4m3 mma.sync (m16n8k32, fp32 accumulate), measured at
//    ~2.3 PFLOP/s on GB300 - well above what decode-sized T needs to stay on
//    the HBM roofline; no operand conversion is needed.  Each 128-wide K block
//    (one scale block) is accumulated in fresh registers and then promoted:
//    acc += blk * (sx * sw).  The scales of the next k-block are fetched while
//    the current one computes.
//  * TMA (cp.async.bulk.tensor, 128-byte swizzle) producer warp + mbarrier
//    ring + eight consumer warps, stream-K over (tile, k-block) iterations.
//    Partial tiles are reduced by the last-arriving CTA in ascending CTA
//    order, so the fp32 result does not depend on timing: the packed-scale
//    and fp32-scale calls produce identical bits.
//  * The scale format only changes how sx is decoded: packed byte
//    ((g*P + kb/4)*Ta + t)*4 + kb%4 -> 2^(u-127), or the fp32 value.
#include <cstdlib>
#include <cstring>

#include "fq_common.cuh"

namespace fq {

namespace es {
constexpr int kBK = 128;
constexpr int kMaxGrid = 1024;

// MT tokens per tile, CW consumer warps of 16 weight rows (BN = 16 * CW, a
// divisor of the 128-wide weight-scale block), one producer warp.
template <int MT, int CW>
struct Cfg {
  static constexpr int NT = MT / 8;
  static constexpr int BN = 16 * CW;
  static constexpr int THREADS = (CW + 1) * 32;
  static constexpr int W_BYTES = BN * kBK;
  static constexpr int X_BYTES = MT * kBK;
  static constexpr int STAGE = W_BYTES + X_BYTES;  // multiple of 1024
  static constexpr int EPI = BN * MT * 2;
  static constexpr int SCALES = (MT + 4) * 4;      // per stage: MT token scale words + sw
  // ~200 KB of weights in flight per SM to cover loaded HBM latency
  static constexpr int STAGES_FIT = (212 * 1024 - EPI - 4096) / (STAGE + SCALES);
  static constexpr int STAGES = STAGES_FIT > 24 ? 24 : STAGES_FIT;
  static constexpr int SLOT = BN * MT;             // fp32 per slot
  static constexpr int SMEM = STAGES * STAGE + EPI + STAGES * SCALES + 2 * STAGES * 8 + 64 + 1024;
  static_assert(STAGES >= 3, "pipeline too shallow");
  static_assert(128 % BN == 0, "tile must sit inside one weight-scale block");
};

struct Problem {
  int T, G, D, N, KB, NB, TT, P, Ta;
  int64_t total;
  const void* sx;
  int fmt;
  const float* sw;
  uint16_t* y;
  float* slots;
  uint32_t* counters;
  uint32_t* err;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mma_e4m3(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
  return s == 0 ? v.x : (s == 1 ? v.y : (s == 2 ? v.z : v.w));
}

// 4-byte asynchronous copy global -> shared (completion tracked by the
// executing thread's cp.async group, announced on an mbarrier below).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (no pending-count increment: the barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Decoded activation scale from its stored word: a packed UE8M0 word holds
// four k-blocks' exponent bytes, byte u meaning 2^(u-127) (u = 0 is the
// subnormal 2^-127, kept exact so both formats give identical bits); an fp32
// word is the scale itself.  `sel` picks byte kb % 4, zero-extended.
template <int FMT>
__device__ __forceinline__ float decode_sx(uint32_t w, uint32_t sel) {
  if (FMT == FQ_SCALE_UE8M0_PACKED) {
    const uint32_t u = __byte_perm(w, 0u, sel);
    return __uint_as_float(u ? (u << 23) : 0x00400000u);
  }
  return __uint_as_float(w);
}

// Fragment row g (0..7) of a 16-row block reads shared-memory row R(g), so the
// two rows of each quarter-warp phase of a 16-byte ld.shared fall in different
// halves of the 128-byte swizzle atom (conflict-free).
__device__ __forceinline__ int frag_row(int g) { return (g >> 1) | ((g & 1) << 2); }

// CTA whose stream-K range holds iteration i: the largest c with rb[c] <= i.
__device__ __forceinline__ int cta_of(const int* rb, int G, int i) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (rb[mid] <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// tile = (g * NB + nb) * TT + tt, NB = N / BN
struct ETile {
  int g, nb, tt;
};
__device__ __forceinline__ ETile etile(const Problem& p, int tile) {
  ETile t;
  const int q = tile / p.TT;
  t.tt = tile - q * p.TT;
  t.g = q / p.NB;
  t.nb = q - t.g * p.NB;
  return t;
}

template <int MT, int CW, int FMT>
__global__ void __launch_bounds__(Cfg<MT, CW>::THREADS, 1)
    fp8_einsum_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, Problem p) {
  using C = Cfg<MT, CW>;
  constexpr int NT = C::NT, S = C::STAGES, BN = C::BN, kCW = CW, kThreads = C::THREADS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint16_t* epi = reinterpret_cast<uint16_t*>(smem + S * C::STAGE);
  uint32_t* scl = reinterpret_cast<uint32_t*>(smem + S * C::STAGE + C::EPI);  // [S][MT + 4]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::STAGE + C::EPI + S * C::SCALES);
  uint64_t* empty = full + S;
  __shared__ int s_flag, s_issued, s_consumed;
  __shared__ volatile int s_abort;
  __shared__ int rb[kMaxGrid + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1 + 32);  // producer's expect-tx arrival + 32 scale-copy arrivals
      mbar_init(&empty[i], kCW);
    }
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_abort = 0;
  }
  if (warp == kCW && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  const int G = gridDim.x, b = blockIdx.x;
  for (int c = tid; c <= G; c += kThreads) rb[c] = int(int64_t(c) * p.total / G);
  __syncthreads();
  const int begin = rb[b], end = rb[b + 1];
  const int KB = p.KB;
  const int NB128 = p.N / 128;

  if (warp == kCW) {
    // ------------------------------------------------ producer warp (all lanes)
    if (end > begin) {
      // weights streamed once (one token tile): evict-first; else keep for reuse
      const uint64_t pol_w = p.TT > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int n_it = end - begin;
      const int npre = n_it < S ? n_it : S;
      if (lane == 0) {  // weights do not depend on the previous kernel: issue them first
        int tile = begin / KB, kb = begin - tile * KB;
        ETile t = etile(p, tile);
        for (int r = 0; r < npre; ++r) {
          mbar_arrive_expect_tx(&full[r], C::STAGE);
          tma_load_2d(stages + r * C::STAGE, &tmW, &full[r], kb * kBK, t.g * p.N + t.nb * BN, pol_w);
          if (++kb == KB && r + 1 < npre) {
            kb = 0;
            t = etile(p, ++tile);
          }
        }
      }
      pdl_wait();
      int tile = begin / KB, kb = begin - tile * KB;
      ETile t = etile(p, tile);
      int issued = 0;
      for (int r = 0; r < n_it; ++r) {
        const int s = r % S;
        if (r >= npre) {
          int ok = 1;
          if (lane == 0) ok = (!s_abort && mbar_wait(&empty[s], uint32_t((r / S - 1) & 1))) ? 1 : 0;
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) {
            if (lane == 0) {
              if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
              s_abort = 1;
            }
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], C::STAGE);
            tma_load_2d(stages + s * C::STAGE, &tmW, &full[s], kb * kBK, t.g * p.N + t.nb * BN, pol_w);
          }
        }
        if (lane == 0)
          tma_load_2d(stages + s * C::STAGE + C::W_BYTES, &tmX, &full[s], t.g * p.D + kb * kBK, t.tt * MT, pol_x);
        // this stage's token scale words and the tile's weight-block scale
        uint32_t* sc = scl + s * (MT + 4);
        if (lane == 0) cp_async4(sc + MT, p.sw + (int64_t(t.g) * KB + kb) * NB128 + (t.nb * BN) / 128);
        if (FMT == FQ_SCALE_UE8M0_PACKED) {
          // packed words of 4 consecutive tokens are contiguous and 16-byte
          // aligned (the token dimension is padded to a multiple of 4)
          for (int c4 = lane; c4 < MT / 4; c4 += 32) {
            const int tok0 = t.tt * MT + 4 * c4;
            if (tok0 < p.Ta)
              cp_async16(sc + 4 * c4,
                         static_cast<const int32_t*>(p.sx) + (int64_t(t.g) * p.P + (kb >> 2)) * p.Ta + tok0);
          }
        } else {
          for (int m = lane; m < MT; m += 32) {
            const int tok = t.tt * MT + m;
            if (tok < p.T)  // tokens past T are not copied; consumers use 0 for them
              cp_async4(sc + m, static_cast<const float*>(p.sx) + (int64_t(tok) * p.G + t.g) * KB + kb);
          }
        }
        cp_async_arrive_noinc(&full[s]);
        ++issued;
        if (++kb == KB && r + 1 < n_it) {
          kb = 0;
          t = etile(p, ++tile);
        }
      }
      if (lane == 0) s_issued = issued;
    }
  } else {
    pdl_wait();
    // Let the next kernel launch only once this one's inputs are final: a
    // dependent may prefetch weights before its own wait, which is safe only
    // if every earlier kernel has finished.
    pdl_launch_dependents();
    const int gq = lane >> 2, c = lane & 3;
    const int rg = frag_row(gq);
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[j][r] = 0.f;
    const uint32_t sbase = smem_u32(stages);
    const uint32_t rowW0 = uint32_t((16 * warp + rg) * kBK), rowW1 = rowW0 + 8 * kBK;
    int tile = begin / KB, kb = begin - tile * KB;
    ETile t = etile(p, tile);
    int seg_kb0 = kb;
    bool first_seg = true;
    int consumed = 0;
    const int n_it = end - begin;
    for (int r = 0; r < n_it; ++r) {
      const int s = r % S;
      bool ok = !s_abort && mbar_wait(&full[s], uint32_t((r / S) & 1));
      if (!ok) {
        if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
        s_abort = 1;
      }
      if (ok) {
        const uint32_t st = sbase + uint32_t(s * C::STAGE);
        // one fp32 chain per 64-byte half when there are few token tiles
        constexpr int NB2 = NT <= 2 ? 2 : 1;
        float blk[NB2][NT][4];
#pragma unroll
        for (int a = 0; a < NB2; ++a)
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) blk[a][j][rr] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t q = uint32_t(((4 * h + c) ^ rg) << 4);
          const uint4 wa = lds128(st + rowW0 + q);
          const uint4 wb = lds128(st + rowW1 + q);
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint4 xv = lds128(st + C::W_BYTES + uint32_t((8 * j + rg) * kBK) + q);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
              mma_e4m3(blk[h % NB2][j], word_of(wa, 2 * ks), word_of(wb, 2 * ks), word_of(wa, 2 * ks + 1),
                       word_of(wb, 2 * ks + 1), word_of(xv, 2 * ks), word_of(xv, 2 * ks + 1));
          }
        }
        const uint32_t* sc = scl + s * (MT + 4);
        const float swv = __uint_as_float(sc[MT]);
        const uint32_t sel = 0x4440u | uint32_t(kb & 3);  // byte kb % 4 of the word, zero-extended
        float sxs[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ml = 8 * j + frag_row(2 * c + hh);
            sxs[j][hh] = (t.tt * MT + ml < p.T) ? decode_sx<FMT>(sc[ml], sel) : 0.f;
          }
        // The stage was read through the generic proxy (ld.shared); the next
        // TMA write into it goes through the async proxy.  Order the two
        // before handing the stage back, or TMA can overwrite it under the read.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        ++consumed;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const float bsum = NB2 == 2 ? __fadd_rn(blk[0][j][rr], blk[NB2 - 1][j][rr]) : blk[0][j][rr];
            acc[j][rr] = __fmaf_rn(bsum, __fmul_rn(sxs[j][rr & 1], swv), acc[j][rr]);
          }
      }
      if (kb == KB - 1 || r == n_it - 1) {
        const bool whole = (seg_kb0 == 0) && (kb == KB - 1);
        bool do_epi = whole;
        if (!whole) {
          float* my = p.slots + (2 * b + (first_seg ? 0 : 1)) * int64_t(C::SLOT);
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) my[((warp * NT + j) * 4 + rr) * 32 + lane] = acc[j][rr];
          named_bar_sync(1, kCW * 32);
          if (tid == 0) {
            const uint32_t nbk = uint32_t(kb - seg_kb0 + 1);
            const uint32_t old = atom_add_acq_rel_gpu(&p.counters[tile], nbk);
            const int last = (old + nbk == uint32_t(KB)) ? 1 : 0;
            if (last) p.counters[tile] = 0;
            s_flag = last;
          }
          named_bar_sync(1, kCW * 32);
          do_epi = s_flag != 0;
          if (do_epi) {
            // Fixed order: ascending CTA index over every contributor's slot
            // (this CTA's own partial included, read back from its slot), so
            // the fp32 sum does not depend on which CTA arrives last.
            constexpr int U = NT <= 2 ? 8 : (NT <= 4 ? 4 : 2);
            const int c0 = cta_of(rb, G, tile * KB), c1 = cta_of(rb, G, tile * KB + KB - 1);
            float tot[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int rr = 0; rr < 4; ++rr) tot[j][rr] = 0.f;
            for (int cb = c0; cb <= c1; cb += U) {
              float v[U][NT][4];
              bool use[U];
#pragma unroll
              for (int u = 0; u < U; ++u) {
                const int cc = cb + u;
                use[u] = cc <= c1 && rb[cc + 1] != rb[cc];
                const int first_tile = use[u] ? rb[cc] / KB : 0;
                const float* sl = p.slots + (2 * int64_t(cc) + (first_tile == tile ? 0 : 1)) * int64_t(C::SLOT);
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                  for (int rr = 0; rr < 4; ++rr)
                    v[u][j][rr] = use[u] ? __ldcg(sl + ((warp * NT + j) * 4 + rr) * 32 + lane) : 0.f;
              }
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (use[u]) {
#pragma unroll
                  for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) tot[j][rr] = __fadd_rn(tot[j][rr], v[u][j][rr]);
                }
            }
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int rr = 0; rr < 4; ++rr) acc[j][rr] = tot[j][rr];
          }
          named_bar_sync(1, kCW * 32);  // s_flag is rewritten by the next segment
        }
        if (do_epi) {
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int nl = 16 * warp + rg + ((rr & 2) ? 8 : 0);
              const int ml = 8 * j + frag_row(2 * c + (rr & 1));
              epi[ml * BN + nl] = f32_to_bf16_bits(acc[j][rr]);
            }
          named_bar_sync(1, kCW * 32);
          const int n0 = t.nb * BN;
          for (int idx = tid; idx < MT * (BN / 8); idx += kCW * 32) {
            const int ml = idx / (BN / 8), c8 = idx % (BN / 8);
            const int tok = t.tt * MT + ml;
            if (tok < p.T) {
              const uint4 v = *reinterpret_cast<const uint4*>(epi + ml * BN + c8 * 8);
              *reinterpret_cast<uint4*>(p.y + (int64_t(tok) * p.G + t.g) * p.N + n0 + c8 * 8) = v;
            }
          }
          named_bar_sync(1, kCW * 32);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) acc[j][rr] = 0.f;
        first_seg = false;
        seg_kb0 = 0;
      }
      if (++kb == KB) {
        kb = 0;
        t = etile(p, ++tile);
      }
    }
    if (tid == 0) s_consumed = consumed;
  }
  __syncthreads();
  if (tid == 0) {
    for (int r = s_consumed; r < s_issued; ++r) mbar_wait(&full[r % S], uint32_t((r / S) & 1));
  }
}

int pick_mt(int64_t T) { return T <= 8 ? 8 : (T <= 16 ? 16 : (T <= 32 ? 32 : 64)); }

template <int MT, int CW, int FMT>
cudaError_t launch_es1(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid, cudaStream_t s,
                       bool pdl) {
  using Cf = Cfg<MT, CW>;
  auto k = fp8_einsum_kernel<MT, CW, FMT>;
  static uint64_t attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch(k, dim3(grid), dim3(Cf::THREADS), size_t(Cf::SMEM), s, pdl, *tw, *tx, p);
}
// The scale format is a compile-time parameter of the kernel.
template <int MT, int CW>
cudaError_t launch_es(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid, cudaStream_t s,
                      bool pdl) {
  return p.fmt == FQ_SCALE_UE8M0_PACKED ? launch_es1<MT, CW, FQ_SCALE_UE8M0_PACKED>(tw, tx, p, grid, s, pdl)
                                        : launch_es1<MT, CW, FQ_SCALE_FP32>(tw, tx, p, grid, s, pdl);
}
}  // namespace es

size_t ws_fp8_group_einsum(int64_t T, int64_t D, int64_t N, int64_t G) {
  DevInfo d;
  if (device_info(&d) != FQ_OK || T < 0 || D < 0 || N < 0 || G < 0) return 0;
  const int mt = es::pick_mt(T);
  return kCounterBytes + size_t(2) * d.sm_count * 128 * mt * 4;
}

}  // namespace fq

using namespace fq;

extern "C" __attribute__((visibility("default"))) fq_status fp8_group_einsum(const uint8_t* xq, const void* sx, int fmt, int64_t T, int64_t G, int64_t D,
                                      const uint8_t* w_gnd, const float* sw_blk, int64_t N, uint16_t* y, void* ws,
                                      size_t ws_bytes, fq_stream_t stream) {
  if (fmt != FQ_SCALE_UE8M0_PACKED && fmt != FQ_SCALE_FP32) return FQ_ERR_ARG;
  if (T < 0 || G < 0 || D < 0 || N < 0 || D % 128 || N % 128) return FQ_ERR_SHAPE;
  if (T > (int64_t(1) << 24) || G > 4096 || D > 65536 || N > (int64_t(1) << 20) || G * N > (int64_t(1) << 30))
    return FQ_ERR_SHAPE;
  if (T == 0 || G == 0 || N == 0) return FQ_OK;
  if (!xq || !sx || !w_gnd || !sw_blk || !y) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(sx) || !aligned16(w_gnd) || !aligned16(sw_blk) || !aligned16(y))
    return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 0) return cuda_status(cudaMemsetAsync(y, 0, size_t(T) * G * N * 2, s));
  const int mt = es::pick_mt(T);
  const int64_t TT = (T + mt - 1) / mt;
  // Schedule: 128-row tiles split stream-K over one CTA per SM.  The other
  // schedule - 64-row tiles, one whole tile per CTA - measured slower on GB300
  // at every decode size (T = 1..256) and is only taken when forced.
  const int64_t tiles64 = G * (N / 64) * TT;
  bool data_parallel = false;
  // FQ_FORCE_SCHEDULE = dp | streamk overrides the choice (tests and studies)
  if (const char* f = std::getenv("FQ_FORCE_SCHEDULE")) {
    if (!std::strcmp(f, "dp") && tiles64 <= es::kMaxGrid) data_parallel = true;
    if (!std::strcmp(f, "streamk")) data_parallel = false;
  }
  const int bn = data_parallel ? 64 : 128;
  es::Problem p = {};
  p.T = int(T);
  p.G = int(G);
  p.D = int(D);
  p.N = int(N);
  p.KB = int(D / 128);
  p.NB = int(N / bn);
  p.TT = int(TT);
  p.P = int((D / 128 + 3) / 4);
  p.Ta = int((T + 3) / 4 * 4);
  const int64_t tiles = G * p.NB * TT;
  if (tiles > kMaxTiles || tiles * p.KB > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  p.total = tiles * p.KB;
  const size_t need = kCounterBytes + size_t(2) * d.sm_count * 128 * mt * 4;
  if (!ws || ws_bytes < need) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  p.sx = sx;
  p.fmt = fmt;
  p.sw = sw_blk;
  p.y = y;
  p.counters = static_cast<uint32_t*>(ws);
  p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.err = d.err_word;
  CUtensorMap tw_map, tx_map;
  if (!tensor_map_u8_2d(&tw_map, w_gnd, uint64_t(D), uint64_t(G * N), uint64_t(D), es::kBK, uint32_t(bn)) ||
      !tensor_map_u8_2d(&tx_map, xq, uint64_t(G * D), uint64_t(T), uint64_t(G * D), es::kBK, uint32_t(mt)))
    return FQ_ERR_CUDA;
  const CUtensorMap* tw = &tw_map;
  const CUtensorMap* tx = &tx_map;
  const int grid = data_parallel ? int(tiles) : int(p.total < d.sm_count ? p.total : d.sm_count);
  const bool pdl = pdl_enabled();
  cudaError_t e;
  if (data_parallel) {
    switch (mt) {
      case 8: e = es::launch_es<8, 4>(tw, tx, p, grid, s, pdl); break;
      case 16: e = es::launch_es<16, 4>(tw, tx, p, grid, s, pdl); break;
      case 32: e = es::launch_es<32, 4>(tw, tx, p, grid, s, pdl); break;
      default: e = es::launch_es<64, 4>(tw, tx, p, grid, s, pdl); break;
    }
  } else {
    switch (mt) {
      case 8: e = es::launch_es<8, 8>(tw, tx, p, grid, s, pdl); break;
      case 16: e = es::launch_es<16, 8>(tw, tx, p, grid, s, pdl); break;
      case 32: e = es::launch_es<32, 8>(tw, tx, p, grid, s, pdl); break;
      default: e = es::launch_es<64, 8>(tw, tx, p, grid, s, pdl); break;
    }
  }
  return cuda_status(e);
}
