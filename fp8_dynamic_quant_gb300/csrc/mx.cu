// 32-element block-scaled FP8 linear ("Reshaping LLM inference dataflow:
// DeepSeek V4 950" section 2.1: every 32 elements share one 8-bit scale,
// E4M3 payloads).
//
//   Y[m, n] = bf16( sum_k (qx[m,k] 2^ex[m,k/32]) (qw[n,k] 2^ew[n,k/32]) )
//
// GB300 design: the 5th-generation tensor cores apply the block scales
// themselves (tcgen05.mma kind::mxf8f6f4.block_scale, one UE8M0 scale per 32
// K per row of each operand), so nothing is converted or promoted in
// software:
//  * warp 0 lane 0: per 128-K block a TMA tile of 128 weight rows and one of
//    MT tokens (128-byte swizzle, the MMA's K-major operand layout) plus the
//    two 512-byte scale chunks (1-D bulk copies), all counted on one mbarrier;
//  * warp 1: allocates tensor memory; lane 0 copies the scale chunks into
//    tensor memory (tcgen05.cp .32x128b.warpx4) and issues four MMAs
//    (M = 128 weight rows, N = MT tokens, K = 32, scale byte j for K step j),
//    accumulating in fp32 tensor memory over the whole segment;
//  * warps 2..5: epilogue, one weight row per thread: drain the accumulator
//    (two buffers alternate), hand partial tiles over stream-K (fp32 partial
//    sums added by the last CTA in ascending CTA order, so results do not
//    depend on timing) and store bf16 through a staging tile.
// The scale chunks are the blocked layout quant_mxfp8 writes: for 128 rows x
// 128 K, row r's byte for K block b at (r % 32) * 16 + ((r % 128) / 32) * 4 + b % 4.
#include <cstdlib>

#include "fq_common.cuh"

namespace fq {
namespace mxk {

constexpr int kBK = 128;
constexpr int kMaxGrid = 1024;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;

template <int MT>
struct Cfg {
  static constexpr int W_BYTES = 128 * kBK;
  static constexpr int X_BYTES = MT * kBK;
  static constexpr int SF_BYTES = 1024;  // weight chunk, then token chunk
  static constexpr int STAGE = W_BYTES + X_BYTES + SF_BYTES;  // multiple of 1024
  static constexpr int STAGES_FIT = (214 * 1024 - 2048) / STAGE;
  static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
  static constexpr int SLOT = 128 * MT;               // fp32 per partial-sum slot
  static constexpr int SF_COL = 2 * MT;               // tensor memory: 2 accumulators, then 8 columns per stage
  static constexpr int SMEM = STAGES * STAGE + (2 * STAGES + 5) * 8 + 1024;
  static_assert(SF_COL + 8 * STAGES <= int(kTmemCols), "tensor-memory budget");
  static_assert(STAGES >= 3, "pipeline too shallow");
};

struct Problem {
  int M, N, K, KB, m_tiles, n_tiles;
  int ahead;  // stages kept in flight (<= the ring)
  int64_t total;
  const uint8_t* xsf;   // blocked token scales
  const uint8_t* wsf;   // blocked weight scales
  uint16_t* y;
  float* slots;
  uint32_t* counters;
  uint32_t* err;
};

__device__ __forceinline__ int cta_of(const int* rb, int G, int i) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (rb[mid] <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// Scale chunk (32 rows x 16 bytes, no swizzle, 8-row groups 128 bytes apart)
// -> tensor memory: every lane quarter receives the 32 x 128-bit block.
__device__ __forceinline__ void sf_copy(uint32_t taddr, uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(128 >> 4) << 32;  // stride byte offset between 8-row groups
  d |= uint64_t(1) << 46;         // descriptor version
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A and B (K-major), UE8M0
// scales, M = 128, N = n, scale byte `j` of both operands.
__host__ __device__ constexpr uint32_t idesc_mx(int n, int j) {
  return (uint32_t(j) << 4) | (uint32_t(n >> 3) << 17) | (1u << 23) | (uint32_t(128 >> 4) << 24) |
         (uint32_t(j) << 29);
}

__device__ __forceinline__ void umma_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::
          "r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    mx_linear_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, Problem p) {
  using C = Cfg<MT>;
  constexpr int S = C::STAGES, kEpi = kEpiWarps * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::STAGE);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;    // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* done_bar = acc_empty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag, s_issued, s_consumed;
  __shared__ volatile int s_abort;
  __shared__ int rb[kMaxGrid + 1];
  __shared__ __align__(16) uint16_t s_ystage[16 * 128];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_abort = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  const int G = gridDim.x, b = blockIdx.x;
  for (int c = tid; c <= G; c += kThreads) rb[c] = int(int64_t(c) * p.total / G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int begin = rb[b], end = rb[b + 1], n_it = end - begin;
  const int KB = p.KB;
  // tile = n_tile * m_tiles + m_tile
  auto w_row = [&](int tile) { return (tile / p.m_tiles) * 128; };
  auto x_row = [&](int tile) { return (tile % p.m_tiles) * MT; };

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      const uint64_t pol_w = p.m_tiles > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int AH = p.ahead < S ? p.ahead : S;
      const int npre = n_it < AH ? n_it : AH;
      {  // weights and their scales do not depend on the previous kernel
        int tile = begin / KB, kb = begin - tile * KB;
        for (int r = 0; r < npre; ++r) {
          uint8_t* st = smem + r * C::STAGE;
          mbar_arrive_expect_tx(&full[r], C::STAGE);
          tma_load_2d(st, &tmW, &full[r], kb * kBK, w_row(tile), pol_w);
          bulk_load(st + C::W_BYTES + C::X_BYTES, p.wsf + (int64_t(tile / p.m_tiles) * KB + kb) * 512, 512u,
                    &full[r]);
          if (++kb == KB) {
            kb = 0;
            ++tile;
          }
        }
      }
      pdl_wait();
      int tile = begin / KB, kb = begin - tile * KB;
      int issued = 0;
      for (int r = 0; r < n_it; ++r) {
        const int s = r % S;
        uint8_t* st = smem + s * C::STAGE;
        if (r >= npre) {
          // iteration r - AH consumed: at most AH stages in flight, slot s free
          const int rq = r - AH;
          if (s_abort || !mbar_wait(&empty[rq % S], uint32_t((rq / S) & 1))) {
            if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::STAGE);
          tma_load_2d(st, &tmW, &full[s], kb * kBK, w_row(tile), pol_w);
          bulk_load(st + C::W_BYTES + C::X_BYTES, p.wsf + (int64_t(tile / p.m_tiles) * KB + kb) * 512, 512u,
                    &full[s]);
        }
        tma_load_2d(st + C::W_BYTES, &tmX, &full[s], kb * kBK, x_row(tile), pol_x);
        // token tiles start at multiples of 128 rows (MT == 128) or are the only tile (MT < 128)
        bulk_load(st + C::W_BYTES + C::X_BYTES + 512, p.xsf + (int64_t(x_row(tile) / 128) * KB + kb) * 512, 512u,
                  &full[s]);
        ++issued;
        if (++kb == KB) {
          kb = 0;
          ++tile;
        }
      }
      s_issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // The whole warp walks the k-blocks (waits and loop control warp-uniform)
    // and one elected lane issues: one thread issuing with a wait per block
    // cost ~0.3 us of issue overhead per block on GB300.
    const uint32_t sbase = smem_u32(smem);
    int kb = begin % KB, seg_kb0 = kb, seg = -1, consumed = 0, s = 0;
    uint32_t ph = 0;
    for (int r = 0; r < n_it; ++r) {
      const bool seg_start = (kb == seg_kb0);
      const bool seg_end = (kb == KB - 1) || (r == n_it - 1);
      if (seg_start) ++seg;
      bool ok = true;
      if (seg_start && seg >= 2) ok = mbar_wait_or_abort(&acc_empty[seg & 1], uint32_t(((seg >> 1) - 1) & 1), &s_abort);
      if (ok) ok = mbar_wait_or_abort(&full[s], ph, &s_abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (lane == 0) {
          if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t st = sbase + uint32_t(s * C::STAGE);
      const uint32_t sfa = tmem + uint32_t(C::SF_COL + 8 * s), sfb = sfa + 4;
      const uint32_t d = tmem + uint32_t((seg & 1) * MT);
      const uint64_t da = umma_desc_k_sw128(st), db = umma_desc_k_sw128(st + C::W_BYTES);
      if (elect_one()) {
        sf_copy(sfa, st + C::W_BYTES + C::X_BYTES);
        sf_copy(sfb, st + C::W_BYTES + C::X_BYTES + 512);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          umma_mx(d, da + uint64_t(2 * j), db + uint64_t(2 * j), idesc_mx(MT, j), sfa, sfb, (!seg_start || j > 0) ? 1u : 0u);
        umma_commit(&empty[s]);
        if (seg_end) umma_commit(&acc_full[seg & 1]);
      }
      __syncwarp();
      ++consumed;
      if (seg_end) seg_kb0 = 0;
      if (++kb == KB) kb = 0;
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (elect_one()) umma_commit(done_bar);
    __syncwarp();
    const bool dok = mbar_wait(done_bar, 0);
    if (lane == 0) {
      if (!dok) atomicOr(p.err, DEVERR_TIMEOUT);
      s_consumed = consumed;  // stages whose copies are known to have landed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue
    pdl_wait();
    pdl_launch_dependents();
    const int q = warp & 3, nl = 32 * q + lane, etid = tid - 64;
    const uint32_t trow = tmem + (uint32_t(32 * q) << 16);
    int tile = begin / KB, kb = begin - tile * KB, seg_kb0 = kb, seg = -1;
    bool first_seg = true;
    for (int r = 0; r < n_it; ++r) {
      const bool seg_start = (kb == seg_kb0);
      const bool seg_end = (kb == KB - 1) || (r == n_it - 1);
      if (seg_start) ++seg;
      if (seg_end) {
        const int n0 = w_row(tile), m0 = x_row(tile);
        const int rows = min(MT, p.M - m0);
        const bool whole = (seg_kb0 == 0) && (kb == KB - 1);
        bool ok = !s_abort && mbar_wait(&acc_full[seg & 1], uint32_t((seg >> 1) & 1));
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
          if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        }
        tc_fence_after();
        const uint32_t tacc = trow + uint32_t((seg & 1) * MT);
        float* my = p.slots + (2 * int64_t(b) + (first_seg ? 0 : 1)) * C::SLOT + nl;
        if (!whole) {
          // this CTA's partial sums -> its slot [MT tokens][128 rows]
#pragma unroll
          for (int h = 0; h < MT / 16; ++h) {
            uint32_t v[16];
            if (ok) tmem_ld16(tacc + uint32_t(16 * h), v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) my[(16 * h + j) * 128] = ok ? __uint_as_float(v[j]) : 0.0f;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && ok) mbar_arrive(&acc_empty[seg & 1]);
          named_bar_sync(1, kEpi);
          if (etid == 0) {
            const uint32_t nbk = uint32_t(kb - seg_kb0 + 1);
            const uint32_t old = atom_add_acq_rel_gpu(&p.counters[tile], nbk);
            const int last = (old + nbk == uint32_t(KB)) ? 1 : 0;
            if (last) p.counters[tile] = 0;  // every contributor has arrived; ready for the next call
            s_flag = last;
          }
          named_bar_sync(1, kEpi);
        }
        const bool do_epi = whole || s_flag != 0;
        if (do_epi) {
          const int c0 = whole ? 0 : cta_of(rb, G, tile * KB), c1 = whole ? -1 : cta_of(rb, G, tile * KB + KB - 1);
#pragma unroll 1
          for (int h = 0; h < MT / 16; ++h) {
            float acc[16];
            if (whole) {
              uint32_t v[16];
              if (ok) tmem_ld16(tacc + uint32_t(16 * h), v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[j] = ok ? __uint_as_float(v[j]) : 0.0f;
            } else {
              // every contributor's slot, this CTA's own included, added in
              // ascending CTA order; four contributors' loads are in flight at once
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
              for (int cb = c0; cb <= c1; cb += 4) {
                float v[4][16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int cc = cb + u;
                  const bool use = cc <= c1 && rb[cc + 1] != rb[cc];
                  const int first_tile = use ? rb[cc] / KB : tile;
                  const float* sl = p.slots + (2 * int64_t(use ? cc : b) + (first_tile == tile ? 0 : 1)) * C::SLOT +
                                    nl + 16 * h * 128;
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[u][j] = use ? __ldcg(sl + j * 128) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (cb + u <= c1 && rb[cb + u + 1] != rb[cb + u]) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = __fadd_rn(acc[j], v[u][j]);
                  }
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) s_ystage[j * 128 + nl] = f32_to_bf16_bits(acc[j]);
            named_bar_sync(1, kEpi);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int piece = i * kEpi + etid, j = piece >> 4, c8 = piece & 15;
              const int m = 16 * h + j, nn = n0 + 8 * c8;
              if (m < rows && nn < p.N) {
                const uint4 v = *reinterpret_cast<const uint4*>(&s_ystage[j * 128 + 8 * c8]);
                st_global_v4(p.y + int64_t(m0 + m) * p.N + nn, v);
              }
            }
            named_bar_sync(1, kEpi);
          }
        }
        if (whole) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && ok) mbar_arrive(&acc_empty[seg & 1]);
        }
        if (!whole) named_bar_sync(1, kEpi);  // s_flag is rewritten by the next segment
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
  if (tid == 0) {
    for (int r = s_consumed; r < s_issued; ++r) mbar_wait(&full[r % S], uint32_t((r / S) & 1));
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MT>
cudaError_t launch_mx(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid, cudaStream_t s,
                      bool pdl) {
  using C = Cfg<MT>;
  auto k = mx_linear_kernel<MT>;
  static uint64_t attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch(k, dim3(grid), dim3(kThreads), size_t(C::SMEM), s, pdl, *tw, *tx, p);
}

int pick_mt(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }
}  // namespace mxk

size_t ws_mxfp8_linear(int64_t M, int64_t K, int64_t N) {
  DevInfo d;
  if (device_info(&d) != FQ_OK || M < 0 || K < 0 || N < 0) return 0;
  return kCounterBytes + size_t(2) * d.sm_count * 128 * mxk::pick_mt(M) * 4;
}

}  // namespace fq

using namespace fq;

extern "C" __attribute__((visibility("default"))) fq_status mxfp8_linear(const uint8_t* xq, const uint8_t* xsf,
                                                                         int64_t M, int64_t K, const uint8_t* wq,
                                                                         const uint8_t* wsf, int64_t N, uint16_t* y,
                                                                         void* ws, size_t ws_bytes,
                                                                         fq_stream_t stream) {
  if (M < 0 || K < 0 || N < 0 || K % 128 || N % 16) return FQ_ERR_SHAPE;
  if (K > 131072 || N > (int64_t(1) << 24) || M > (int64_t(1) << 24)) return FQ_ERR_SHAPE;
  if (M == 0 || N == 0) return FQ_OK;
  if (!xq || !xsf || !wq || !wsf || !y) return FQ_ERR_NULL;
  if (!aligned16(xq) || !aligned16(xsf) || !aligned16(wq) || !aligned16(wsf) || !aligned16(y)) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, size_t(M) * N * 2, s));
  const int mt = mxk::pick_mt(M);
  mxk::Problem p = {};
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.KB = int(K / 128);
  p.m_tiles = int((M + mt - 1) / mt);
  p.n_tiles = int((N + 127) / 128);
  const int64_t tiles = int64_t(p.m_tiles) * p.n_tiles;
  if (tiles > kMaxTiles || tiles * p.KB > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  p.total = tiles * p.KB;
  const size_t need = kCounterBytes + size_t(2) * d.sm_count * 128 * mt * 4;
  if (!ws || ws_bytes < need) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  p.xsf = xsf;
  p.wsf = wsf;
  p.y = y;
  p.counters = static_cast<uint32_t*>(ws);
  p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.err = d.err_word;
  CUtensorMap tw_map, tx_map;
  if (!tensor_map_u8_2d(&tw_map, wq, uint64_t(K), uint64_t(N), uint64_t(K), mxk::kBK, 128u) ||
      !tensor_map_u8_2d(&tx_map, xq, uint64_t(K), uint64_t(M), uint64_t(K), mxk::kBK, uint32_t(mt)))
    return FQ_ERR_CUDA;
  // at least 4 k-blocks per CTA: a CTA's fixed cost (pipeline fill, epilogue)
  // and a tile's stream-K hand-off grow with the number of CTAs sharing it
  {  // stages in flight: about 120 KB per SM (see the W8A8 GEMM's stage cap)
    const int stage = 128 * 128 + mt * 128 + 1024;
    int ah = (122880 + stage / 2) / stage;
    if (const char* v = std::getenv("FQ_STAGES_AHEAD")) ah = std::atoi(v);
    p.ahead = ah < 2 ? 2 : ah;
  }
  // at least 4 k-blocks a CTA, 8 with 64- or 128-token tiles: a tile's last
  // CTA adds its partners' partial slots (128 x MT fp32 each) on the critical
  // path, so fewer partners pay off once the slots are large (K=4096, N=1024
  // on GB300: M=64 13.7 -> 11.0 us, M=128 23.1 -> 15.9 us)
  const int minb = mt >= 64 ? 8 : 4;
  const int64_t by_work = (p.total + minb - 1) / minb;
  int grid = int(by_work < d.sm_count ? (by_work > 0 ? by_work : 1) : d.sm_count);
  {
    const int g = whole_tile_grid(tiles, d.sm_count);
    if (g > 0 && g <= grid) grid = g;
  }
  const bool pdl = pdl_enabled();
  cudaError_t e;
  switch (mt) {
    case 16: e = mxk::launch_mx<16>(&tw_map, &tx_map, p, grid, s, pdl); break;
    case 32: e = mxk::launch_mx<32>(&tw_map, &tx_map, p, grid, s, pdl); break;
    case 64: e = mxk::launch_mx<64>(&tw_map, &tx_map, p, grid, s, pdl); break;
    default: e = mxk::launch_mx<128>(&tw_map, &tx_map, p, grid, s, pdl); break;
  }
  return cuda_status(e);
}
