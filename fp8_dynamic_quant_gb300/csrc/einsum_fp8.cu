// Block-scaled FP8 grouped einsum, the consumer of the packed UE8M0
// activation scales ("SGLang PR #34277 digest": motivation and
// implementation breakdown item 3 - deep_gemm.fp8_einsum reads the
// TMA-aligned packed scales; packed and fp32 scales must give bit-identical
// outputs).
//
//   Y[t, g, n] = bf16( sum_kb sx[t,g,kb] * sw[g,kb,n/128] * sum_{d in kb} xq[t,g,d] * W[g,d,n] )
//
// GB300 design (5th-generation tensor cores, operands straight from TMA):
//  * Swap-AB tiles: BM weight rows (n; 128 = one weight-scale block, or 64
//    when whole 64-row tiles fill the SMs and 128-row ones do not) x MT
//    tokens (16, 32 or 64; more tokens take several token tiles), one tile
//    per (g, n-block, token tile).  Weights E4M3 [G, N, D] K-major,
//    activations E4M3 [T, G, D]; both land by TMA in the 128-byte-swizzled
//    K-major layout the MMA reads, so nothing is converted.
//  * A pipeline stage holds KD (4, 2 or 1) consecutive K blocks of a tile,
//    fetched by one 3-D TMA box for the weights and one for the activations.
//  * warp 0 lane 0: TMA producer (weights of the first stages are issued at
//    kernel entry, before the wait on the previous kernel);
//  * warp 1: allocates tensor memory; the whole warp walks the stages and
//    one elected lane issues, per 128-wide K block, four tcgen05.mma
//    kind::f8f6f4 (M = BM, N = MT, K = 32) into a fresh fp32 accumulator
//    slot in tensor memory, and commits once per group of four K blocks (two
//    groups of slots alternate);
//  * warps 2..5: one weight row per thread.  Per group they wait once, then
//    per stage drain its slots (tcgen05.ld) and promote them into fp32
//    registers: acc += blk * (sx[t] * sw) - the per-128-K block scaling.  The
//    scales stream in 8-16 blocks ahead by asynchronous copies.
//  * Whole tiles per CTA when they fill the SMs; otherwise stream-K over the
//    flattened (tile, stage) range, one CTA per SM: the partial tiles at a
//    CTA's range ends go to workspace slots and the last CTA to finish a tile
//    adds every contributor's slot in ascending CTA order, so the fp32 result
//    does not depend on timing: the packed-scale and fp32-scale calls produce
//    identical bits, and a token's row does not depend on the other tokens of
//    the call.
//  * The scale format only changes how sx is decoded: packed byte
//    ((g*P + kb/4)*Ta + t)*4 + kb%4 -> 2^(u-127), or the fp32 value.
#include <cstdlib>
#include <cstring>

#include "fq_common.cuh"

namespace fq {

namespace es {
constexpr int kBK = 128;
constexpr int kMaxGrid = 1024;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
// Per-token promotion factors sx[t, kb] * sw[kb] come from a table in shared
// memory filled for up to kTB K blocks of a tile at a time, the next piece
// fetched while the current one is in use: per stage the promotion reads no
// global memory.  (Fetching each stage's scale words by 4-byte asynchronous
// copies in the promotion loop cost ~3 us a call at T = 1 on GB300.)
constexpr int kTB = 32;
// K blocks per tensor-core commit.  A tcgen05.commit added ~80 ns to the
// issuing loop on GB300, more than two decode-sized MMAs (~33 ns each), so
// stage release and the accumulator hand-off are signalled once per group of
// K blocks; a group also ends at every stream-K segment end and at the end of
// the CTA's range.
constexpr int kGroupBars = 24;  // ring of group-completion barriers (more than the stages)
// Blocks per commit group (two groups of MT-column slots in tensor memory).
template <int MT>
struct GroupSize {
  static constexpr int value = 4;
};

// Walks a CTA's (tile, K block) iterations and their commit groups; every
// role keeps one, so they agree on the group boundaries.
template <int GROUP>
struct GroupCursor {
  int r = 0, kb = 0, g = 0, cnt = 0;
  // is iteration r the last of its group?
  __device__ __forceinline__ bool group_end(int KB, int n_it) const {
    return cnt + 1 == GROUP || kb == KB - 1 || r == n_it - 1;
  }
  __device__ __forceinline__ void advance(int KB, int n_it) {
    if (group_end(KB, n_it)) {
      ++g;
      cnt = 0;
    } else {
      ++cnt;
    }
    if (++kb == KB) kb = 0;
    ++r;
  }
  // Chunk steps (KD blocks, KD dividing GROUP, KB and n_it; groups start at
  // chunk starts, so no group ends inside a chunk): does the chunk at the
  // cursor end its group, and the step past it.
  __device__ __forceinline__ bool chunk_ends_group(int KD, int KB, int n_it) const {
    return cnt + KD == GROUP || kb + KD == KB || r + KD == n_it;
  }
  __device__ __forceinline__ void advance_chunk(int KD, int KB, int n_it) {
    if (chunk_ends_group(KD, KB, n_it)) {
      ++g;
      cnt = 0;
    } else {
      cnt += KD;
    }
    kb += KD;
    if (kb == KB) kb = 0;
    r += KD;
  }
};

// BM weight rows per tile: 128 (tcgen05 M = 128) or 64 (M = 64; the
// accumulator's row r then sits in tensor-memory lane 32 * (r / 16) + r % 16,
// the first 16 lanes of each warp's quarter).
template <int MT, int BM>
struct Cfg {
  static constexpr int W_SUB = BM * kBK;  // one K block of the weight tile (multiple of 1024)
  static constexpr int X_SUB = MT * kBK;  // one K block of the token tile (multiple of 1024)
  static constexpr int GROUP = GroupSize<MT>::value;
  static constexpr int NACC = 2 * GROUP;           // accumulator slots: two groups of K blocks
  static constexpr uint32_t TMEM_COLS = NACC * MT <= 128 ? 128u : (NACC * MT <= 256 ? 256u : 512u);
  static constexpr int SLOT = BM * MT;              // fp32 per partial-sum slot
  static_assert(NACC * MT <= 512, "tensor-memory budget");
  static_assert(GROUP % 4 == 0, "a commit group holds whole stages (KD divides 4)");
};
// A stage holds KD consecutive K blocks (1, 2 or 4) of one tile: KD weight
// sub-tiles, then KD token sub-tiles, each fetched by one 3-D TMA box.  TMA
// throughput per SM is set by the number of copies more than by their bytes
// (measured on GB300 with one CTA per SM streaming 256 MB: 8 KB boxes 3.3 TB/s,
// 16 KB 6.0, 32-64 KB 6.2-6.4), so small tiles fetch several K blocks at once.
constexpr int kStageBudget = 200 * 1024;  // ~200 KB of stages in flight per SM (beside the factor table)
constexpr int kMaxStages = 16;
constexpr int kMinStages = 4;
static_assert(kGroupBars > kMaxStages, "group barriers must outnumber the stages (no parity aliasing)");
__host__ __device__ constexpr int stage_bytes(int KD, int BM, int MT) { return KD * (BM + MT) * kBK; }
__host__ __device__ constexpr int smem_bytes(int S, int stage) { return S * stage + (S + kGroupBars + 3) * 8 + 1024; }

struct Problem {
  int T, G, D, N, KB, NB, TT, P, Ta;
  int NS;     // weight-scale blocks along N (N / 128); NB counts tiles of BM rows
  int KD;     // K blocks per stage (divides KB)
  int S;      // stages in the ring
  int stage;  // bytes per stage
  int ahead;  // stages kept in flight (<= S)
  int pre_w;  // weight chunks issued before the wait on the previous kernel (0: all of `ahead`)
  int64_t total;  // stream-K units: (tile, chunk of KD K blocks) pairs
  const void* sx;
  const float* sw;
  uint16_t* y;
  float* slots;
  uint32_t* counters;
  uint32_t* err;
};

// First K-block iteration of CTA c's stream-K range: the ranges split the
// (tile, chunk) units evenly, floor(c * total / G) chunks of KD blocks each.
__device__ __forceinline__ int range_begin(const Problem& p, int G, int c) {
  return int(int64_t(c) * p.total / G) * p.KD;
}
// CTA whose stream-K range holds K-block iteration i: the largest c with range_begin(c) <= i.
__device__ __forceinline__ int cta_of(const Problem& p, int G, int i) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (range_begin(p, G, mid) <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// tile = (g * NB + nb) * TT + tt
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

// Activation scale of K block kb from its stored word: a packed UE8M0 word
// holds four K blocks' exponent bytes, byte u meaning 2^(u-127) (u = 0 is the
// subnormal 2^-127, kept exact so both formats give identical bits); an fp32
// word is the scale itself.
template <int FMT>
__device__ __forceinline__ float decode_sx(uint32_t w, int kb) {
  if (FMT == FQ_SCALE_UE8M0_PACKED) {
    const uint32_t u = (w >> (8 * (kb & 3))) & 0xFFu;
    return __uint_as_float(u ? (u << 23) : 0x00400000u);
  }
  return __uint_as_float(w);
}

// 4-byte asynchronous copy global -> shared, tracked by the issuing thread's
// commit groups.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (E4M3 x E4M3 -> fp32), one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4: fp32 accumulator (bits 4-5 = 1),
// A and B E4M3 (format 0) and K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f8(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

template <int MT, int FMT, int BM>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_einsum_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, Problem p) {
  using C = Cfg<MT, BM>;
  constexpr int kEpi = kEpiWarps * 32;
  const int S = p.S, KD = p.KD, STAGE = p.stage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* grp = full + S;                 // [kGroupBars]: the MMAs of group g have completed
  uint64_t* acc_empty = grp + kGroupBars;   // [2]: the epilogue has drained group g's slots
  uint64_t* done_bar = acc_empty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_flag, s_issued, s_consumed;
  __shared__ volatile int s_abort;
  __shared__ __align__(16) float s_tab[2][kTB * MT];  // promotion factors [piece buffer][block][token]
  __shared__ float s_tsw[2][kTB];                     // weight-block scales of the piece
  __shared__ __align__(16) uint16_t s_ystage[16 * BM];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  int npre = 0;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    for (int i = 0; i < kGroupBars; ++i) mbar_init(&grp[i], 1);
    for (int i = 0; i < 2; ++i) mbar_init(&acc_empty[i], kEpiWarps);
    mbar_init(done_bar, 1);
    fence_barrier_init();
    s_issued = 0;
    s_consumed = 0;
    s_abort = 0;
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    // weights do not depend on the previous kernel: the first stages go out now
    const int b0 = range_begin(p, G, b), b1 = range_begin(p, G, b + 1);
    npre = min((b1 - b0) / KD, p.ahead);
    if (p.pre_w > 0 && p.pre_w < npre) npre = p.pre_w;
    const uint64_t pol_w = p.TT > 1 ? policy_evict_normal() : policy_evict_first();
    int tile = b0 / p.KB, kb = b0 - tile * p.KB;
    ETile t = etile(p, tile);
    for (int q = 0; q < npre; ++q) {
      mbar_arrive_expect_tx(&full[q], STAGE);
      tma_load_3d(smem + q * STAGE, &tmW, &full[q], 0, t.g * p.N + t.nb * BM, kb, pol_w);
      kb += KD;
      if (kb == p.KB && q + 1 < npre) {
        kb = 0;
        t = etile(p, ++tile);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int begin = range_begin(p, G, b), end = range_begin(p, G, b + 1), n_it = end - begin;
  const int KB = p.KB;

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      const uint64_t pol_w = p.TT > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      pdl_wait();
      int tile = begin / KB, kb = begin - tile * KB;
      ETile t = etile(p, tile);
      int issued = 0;
      GroupCursor<C::GROUP> lag;  // at chunk q - ahead, whose group gates the refill
      lag.kb = kb;
      const int nq = n_it / KD;
      // chunks [npre_w, npre_all) of the first lap go out right after the wait,
      // into ring slots not yet used; from npre_all on a group must complete
      const int npre_all = min(nq, p.ahead);
      const int npre_w = (p.pre_w > 0 && p.pre_w < npre_all) ? p.pre_w : npre_all;
      for (int q = 0, s = 0; q < nq; ++q) {
        uint8_t* st = smem + s * STAGE;
        if (q >= npre_w && q < npre_all) {
          mbar_arrive_expect_tx(&full[s], STAGE);
          tma_load_3d(st, &tmW, &full[s], 0, t.g * p.N + t.nb * BM, kb, pol_w);
        } else if (q >= npre_all) {
          // the group holding chunk q - ahead completed: at most `ahead`
          // stages in flight, and (q - S <= q - ahead) stage s is free
          if (q > p.ahead) lag.advance_chunk(KD, KB, n_it);
          const int gl = lag.g;
          if (!mbar_wait_or_abort(&grp[gl % kGroupBars], uint32_t((gl / kGroupBars) & 1), &s_abort)) {
            if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
            s_abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[s], STAGE);
          tma_load_3d(st, &tmW, &full[s], 0, t.g * p.N + t.nb * BM, kb, pol_w);
        }
        tma_load_3d(st + KD * C::W_SUB, &tmX, &full[s], 0, t.tt * MT, t.g * KB + kb, pol_x);
        ++issued;
        if (++s == S) s = 0;
        kb += KD;
        if (kb == KB && q + 1 < nq) {
          kb = 0;
          t = etile(p, ++tile);
        }
      }
      s_issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    // The whole warp walks the chunks (waits and loop control warp-uniform)
    // and one elected lane issues a chunk's KD x 4 MMAs as one straight
    // sequence from a base descriptor plus constant offsets (16-byte units in
    // the low field).  Measured on GB300 with decode-sized MMAs: ~30 ns per
    // MMA this way, against ~110 ns when one thread issued block by block
    // with a wait between blocks.
    const uint64_t da0 = umma_desc_k_sw128(smem_u32(smem));
    const uint64_t db0 = umma_desc_k_sw128(smem_u32(smem) + uint32_t(KD * C::W_SUB));
    constexpr uint32_t idesc = idesc_f8(BM, MT);
    int consumed = 0, s = 0;
    uint32_t phase = 0;
    GroupCursor<C::GROUP> cur;
    cur.kb = begin % KB;
    const int nq = n_it / KD;
    for (int qi = 0; qi < nq; ++qi) {
      bool ok = true;
      // a group starts with this chunk and reuses the slots of the group two back
      if (cur.cnt == 0 && cur.g >= 2)
        ok = mbar_wait_or_abort(&acc_empty[cur.g & 1], uint32_t(((cur.g >> 1) - 1) & 1), &s_abort);
      if (ok) ok = mbar_wait_or_abort(&full[s], phase, &s_abort);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (lane == 0) {
          if (!s_abort) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const uint64_t so = uint64_t(uint32_t(s * STAGE) >> 4);
      const uint64_t da = da0 + so, db = db0 + so;
      const uint32_t d = tmem + uint32_t(((cur.g & 1) * C::GROUP + cur.cnt) * MT);
      const bool gend = cur.chunk_ends_group(KD, KB, n_it);
      if (elect_one()) {
#pragma unroll
        for (int kd = 0; kd < 4; ++kd) {
          if (kd < KD) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              umma_f8(d + uint32_t(kd * MT), da + uint64_t((kd * C::W_SUB) >> 4) + uint64_t(2 * j),
                      db + uint64_t((kd * C::X_SUB) >> 4) + uint64_t(2 * j), idesc, j > 0 ? 1u : 0u);
          }
        }
        // one commit per group: releases the group's stages and hands its slots to the epilogue
        if (gend) umma_commit(&grp[cur.g % kGroupBars]);
      }
      __syncwarp();
      cur.advance_chunk(KD, KB, n_it);
      ++consumed;
      if (++s == S) {
        s = 0;
        phase ^= 1u;
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
    // ------------------------------------------------ promotion + epilogue
    pdl_wait();
    // Let the next kernel launch only once this one's inputs are final: a
    // dependent may prefetch weights before its own wait, which is safe only
    // if every earlier kernel has finished.
    pdl_launch_dependents();
    // this thread's weight row of the tile (BM = 64: lanes 0-15 of each quarter)
    const int q = warp & 3, etid = tid - 64;
    const bool rowv = BM == 128 || lane < 16;
    const int nl = BM == 128 ? 32 * q + lane : 16 * q + (lane & 15);
    const uint32_t trow = tmem + (uint32_t(32 * q) << 16);
    float acc[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[j] = 0.0f;
    int tile = begin / KB, kb = begin - tile * KB, seg_kb0 = kb;
    ETile t = etile(p, tile);
    bool first_seg = true;
    // Promotion factors, a piece (<= kTB blocks of one tile) at a time:
    // every epilogue thread copies a share of the piece's stored scale words
    // and weight-block scales into a table buffer (4-byte asynchronous
    // copies), then, after a barrier, turns its share into sx * sw in place.
    auto fetch = [&](int buf, int tile_f, int kb_f, int len) {
      const ETile tp = etile(p, tile_f);
      uint32_t* tw = reinterpret_cast<uint32_t*>(s_tab[buf]);
      for (int idx = etid; idx < len * MT; idx += kEpi) {
        const int kbi = idx / MT, m = idx - kbi * MT, tok = tp.tt * MT + m, kbb = kb_f + kbi;
        if (tok < p.T) {
          const void* src = FMT == FQ_SCALE_UE8M0_PACKED
                                ? static_cast<const void*>(static_cast<const uint32_t*>(p.sx) +
                                                           (int64_t(tp.g) * p.P + (kbb >> 2)) * p.Ta + tok)
                                : static_cast<const void*>(static_cast<const float*>(p.sx) +
                                                           (int64_t(tok) * p.G + tp.g) * KB + kbb);
          cp_async4(tw + idx, src);
        }
      }
      for (int idx = etid; idx < len; idx += kEpi)
        cp_async4(&s_tsw[buf][idx], p.sw + (int64_t(tp.g) * KB + kb_f + idx) * p.NS + (tp.nb * BM) / 128);
      cp_async_commit();
    };
    auto convert = [&](int buf, int tile_f, int kb_f, int len) {
      cp_async_wait<0>();  // this thread's copies of the piece (nothing was committed after them)
      named_bar_sync(1, kEpi);
      const ETile tp = etile(p, tile_f);
      const uint32_t* tw = reinterpret_cast<const uint32_t*>(s_tab[buf]);
      for (int idx = etid; idx < len * MT; idx += kEpi) {
        const int kbi = idx / MT, m = idx - kbi * MT, tok = tp.tt * MT + m;
        const float f = tok < p.T ? __fmul_rn(decode_sx<FMT>(tw[idx], kb_f + kbi), s_tsw[buf][kbi]) : 0.0f;
        s_tab[buf][idx] = f;
      }
      named_bar_sync(1, kEpi);
    };
    // blocks of the piece starting at (tile, kb) with `left` blocks left in the range
    auto piece_len = [&](int kb_f, int left) { return min(min(kTB - kb_f % kTB, KB - kb_f), left); };
    const int nq = n_it / KD;
    int pbuf = 0, pc_kb0 = kb;
    if (nq > 0) fetch(0, tile, kb, piece_len(kb, n_it));
    // tensor-memory loads in flight at once: 64 registers' worth of blocks
    constexpr int LB = 64 / MT;
    GroupCursor<C::GROUP> ec;
    ec.kb = kb;
    bool gok = true;
    for (int qi = 0; qi < nq; ++qi) {
      const bool seg_end = (kb + KD == KB) || (qi == nq - 1);
      if (qi == 0 || kb % kTB == 0) {
        // a piece starts: its factors are ready once converted; the next
        // piece's scales go out now (its buffer's previous piece is done)
        if (qi > 0) pbuf ^= 1;
        const int left = n_it - qi * KD, len = piece_len(kb, left);
        pc_kb0 = kb;
        convert(pbuf, tile, kb, len);
        if (len < left) {
          const int kb_n = kb + len == KB ? 0 : kb + len, tile_n = kb + len == KB ? tile + 1 : tile;
          fetch(pbuf ^ 1, tile_n, kb_n, piece_len(kb_n, left - len));
        }
      }
      const float* sf = s_tab[pbuf] + (kb - pc_kb0) * MT;
      if (ec.cnt == 0) {  // a group starts: wait once for all of its MMAs
        gok = mbar_wait_or_abort(&grp[ec.g % kGroupBars], uint32_t((ec.g / kGroupBars) & 1), &s_abort);
        gok = __all_sync(0xFFFFFFFFu, gok);
        if (!gok) {
          if (!s_abort && lane == 0) atomicOr(p.err, DEVERR_TIMEOUT);
          s_abort = 1;
        }
        tc_fence_after();
      }
      const bool ok = gok;
      if (ok) {
        // up to LB blocks' accumulators loaded together, one wait, then
        // promoted in order: acc += blk * f
#pragma unroll
        for (int kd0 = 0; kd0 < 4; kd0 += LB) {
          if (kd0 < KD) {
            uint32_t v[LB][MT / 16][16];
#pragma unroll
            for (int u = 0; u < LB; ++u) {
              if (kd0 + u < KD) {
                const uint32_t acol = uint32_t(((ec.g & 1) * C::GROUP + ec.cnt + kd0 + u) * MT);
#pragma unroll
                for (int h = 0; h < MT / 16; ++h) tmem_ld16(trow + acol + uint32_t(16 * h), v[u][h]);
              }
            }
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < LB; ++u) {
              if (kd0 + u < KD) {
                const float* fk = sf + (kd0 + u) * MT;
#pragma unroll
                for (int j4 = 0; j4 < MT / 4; ++j4) {
                  const float4 f = *reinterpret_cast<const float4*>(fk + 4 * j4);
                  float* a4 = acc + 4 * j4;
                  const uint32_t* v4 = &v[u][j4 >> 2][4 * (j4 & 3)];
                  a4[0] = __fmaf_rn(__uint_as_float(v4[0]), f.x, a4[0]);
                  a4[1] = __fmaf_rn(__uint_as_float(v4[1]), f.y, a4[1]);
                  a4[2] = __fmaf_rn(__uint_as_float(v4[2]), f.z, a4[2]);
                  a4[3] = __fmaf_rn(__uint_as_float(v4[3]), f.w, a4[3]);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      // the group's last chunk is read: its slots may take the group after next
      if (ec.chunk_ends_group(KD, KB, n_it) && lane == 0 && ok) mbar_arrive(&acc_empty[ec.g & 1]);
      ec.advance_chunk(KD, KB, n_it);
      __syncwarp();  // sf is rewritten for the next chunk
      if (seg_end) {
        // ---- segment end: tile `tile`, K blocks [seg_kb0, kb + KD - 1]
        const int n0 = t.nb * BM, m0 = t.tt * MT;
        const int rows = min(MT, p.T - m0);
        const bool whole = (seg_kb0 == 0) && (kb + KD == KB);
        if (!whole) {
          // this CTA's partial sums -> its slot [MT tokens][BM rows]
          float* my = p.slots + (2 * int64_t(b) + (first_seg ? 0 : 1)) * C::SLOT + nl;
          if (rowv) {
#pragma unroll
            for (int j = 0; j < MT; ++j) my[j * BM] = acc[j];
          }
          named_bar_sync(1, kEpi);
          if (etid == 0) {
            const uint32_t nbk = uint32_t(kb + KD - seg_kb0);
            const uint32_t old = atom_add_acq_rel_gpu(&p.counters[tile], nbk);
            const int last = (old + nbk == uint32_t(KB)) ? 1 : 0;
            if (last) p.counters[tile] = 0;  // every contributor has arrived; ready for the next call
            s_flag = last;
          }
          named_bar_sync(1, kEpi);
        }
        const bool do_epi = whole || s_flag != 0;
        if (do_epi) {
          if (!whole) {
            // every contributor's slot, this CTA's own included, added in
            // ascending CTA order; four contributors' loads in flight at once
            const int c0 = cta_of(p, G, tile * KB), c1 = cta_of(p, G, tile * KB + KB - 1);
#pragma unroll
            for (int j = 0; j < MT; ++j) acc[j] = 0.0f;
            for (int cb = c0; cb <= c1; cb += 4) {
#pragma unroll
              for (int h = 0; h < MT / 16; ++h) {
                float vv[4][16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int cc = cb + u;
                  const int cb0 = range_begin(p, G, cc);
                  const bool use = cc <= c1 && range_begin(p, G, cc + 1) != cb0;
                  const int first_tile = use ? cb0 / KB : tile;
                  const float* sl = p.slots + (2 * int64_t(use ? cc : b) + (first_tile == tile ? 0 : 1)) * C::SLOT +
                                    nl + 16 * h * BM;
#pragma unroll
                  for (int j = 0; j < 16; ++j) vv[u][j] = (use && rowv) ? __ldcg(sl + j * BM) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (cb + u <= c1 && range_begin(p, G, cb + u + 1) != range_begin(p, G, cb + u)) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[16 * h + j] = __fadd_rn(acc[16 * h + j], vv[u][j]);
                  }
              }
            }
          }
          // bf16 through a staging tile, 16 tokens at a time, 16-byte stores
#pragma unroll
          for (int h = 0; h < MT / 16; ++h) {
            if (rowv) {
#pragma unroll
              for (int j = 0; j < 16; ++j) s_ystage[j * BM + nl] = f32_to_bf16_bits(acc[16 * h + j]);
            }
            named_bar_sync(1, kEpi);
            // 16 tokens x BM / 8 chunks of 8 outputs: one or two 16-byte stores a thread
#pragma unroll
            for (int i = 0; i < BM / 64; ++i) {
              const int piece = i * kEpi + etid, j = piece / (BM / 8), c8 = piece % (BM / 8);
              const int m = 16 * h + j;
              if (m < rows)
                st_global_v4(p.y + (int64_t(m0 + m) * p.G + t.g) * p.N + n0 + 8 * c8,
                             *reinterpret_cast<const uint4*>(&s_ystage[j * BM + 8 * c8]));
            }
            named_bar_sync(1, kEpi);
          }
        }
        if (!whole) named_bar_sync(1, kEpi);  // s_flag is rewritten by the next segment
#pragma unroll
        for (int j = 0; j < MT; ++j) acc[j] = 0.0f;
        first_seg = false;
        seg_kb0 = 0;
      }
      kb += KD;
      if (kb == KB) {
        kb = 0;
        t = etile(p, ++tile);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    for (int r = s_consumed; r < s_issued; ++r) mbar_wait(&full[r % S], uint32_t((r / S) & 1));
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

int pick_mt(int64_t T) { return T <= 16 ? 16 : (T <= 32 ? 32 : 64); }

template <int MT, int FMT, int BM>
cudaError_t launch_es1(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int grid, cudaStream_t s,
                       bool pdl) {
  auto k = fp8_einsum_kernel<MT, FMT, BM>;
  static uint64_t attr_done = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_done & (1ull << (dev & 63)))) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes(kMaxStages, kStageBudget / kMaxStages));
    if (e != cudaSuccess) return e;
    attr_done |= 1ull << (dev & 63);
  }
  return launch(k, dim3(grid), dim3(kThreads), size_t(smem_bytes(p.S, p.stage)), s, pdl, *tw, *tx, p);
}
// The scale format is a compile-time parameter of the kernel.
template <int MT>
cudaError_t launch_es(const CUtensorMap* tw, const CUtensorMap* tx, const Problem& p, int fmt, int bm, int grid,
                      cudaStream_t s, bool pdl) {
  if (bm == 64)
    return fmt == FQ_SCALE_UE8M0_PACKED ? launch_es1<MT, FQ_SCALE_UE8M0_PACKED, 64>(tw, tx, p, grid, s, pdl)
                                        : launch_es1<MT, FQ_SCALE_FP32, 64>(tw, tx, p, grid, s, pdl);
  return fmt == FQ_SCALE_UE8M0_PACKED ? launch_es1<MT, FQ_SCALE_UE8M0_PACKED, 128>(tw, tx, p, grid, s, pdl)
                                      : launch_es1<MT, FQ_SCALE_FP32, 128>(tw, tx, p, grid, s, pdl);
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
  es::Problem p = {};
  p.T = int(T);
  p.G = int(G);
  p.D = int(D);
  p.N = int(N);
  p.KB = int(D / 128);
  p.NS = int(N / 128);
  p.TT = int((T + mt - 1) / mt);
  p.P = int((D / 128 + 3) / 4);
  p.Ta = int((T + 3) / 4 * 4);
  // Tile rows: 128 when whole 128-row tiles fill the SMs; else 64-row tiles
  // (M = 64 MMAs, half the weight bytes per CTA) when those do - whole tiles
  // need no partial-sum hand-off; else 128-row tiles under stream-K.
  int bm = 128;
  {
    const int64_t t128 = G * int64_t(p.NS) * p.TT;
    if (whole_tile_grid(t128, d.sm_count) <= 0 && whole_tile_grid(2 * t128, d.sm_count) > 0) bm = 64;
    if (const char* v = std::getenv("FQ_EINSUM_BM")) bm = std::atoi(v) == 64 ? 64 : 128;
  }
  p.NB = int(N / bm);
  // K blocks per stage: the most of 4, 2, 1 that divides KB and leaves at
  // least kMinStages stages (FQ_EINSUM_KD = 1 | 2 | 4 fixes it for tests)
  {
    int kd = 4;
    while (kd > 1 && (p.KB % kd || es::kStageBudget / es::stage_bytes(kd, bm, mt) < es::kMinStages)) kd >>= 1;
    if (const char* v = std::getenv("FQ_EINSUM_KD")) {
      const int f = std::atoi(v);
      if ((f == 1 || f == 2 || f == 4) && p.KB % f == 0 &&
          es::kStageBudget / es::stage_bytes(f, bm, mt) >= es::kMinStages)
        kd = f;
    }
    p.KD = kd;
    p.stage = es::stage_bytes(kd, bm, mt);
    const int fit = es::kStageBudget / p.stage;
    p.S = fit > es::kMaxStages ? es::kMaxStages : fit;
  }
  const int64_t tiles = G * p.NB * int64_t(p.TT);
  if (tiles > kMaxTiles || tiles * p.KB > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  p.total = tiles * (p.KB / p.KD);
  const size_t need = kCounterBytes + size_t(2) * d.sm_count * 128 * mt * 4;
  if (!ws || ws_bytes < need) return FQ_ERR_WORKSPACE;
  if (!aligned16(ws)) return FQ_ERR_ALIGN;
  p.sx = sx;
  p.sw = sw_blk;
  p.y = y;
  p.counters = static_cast<uint32_t*>(ws);
  p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  p.err = d.err_word;
  // 3-D views (128 bytes of a K block, rows, K blocks): W [G*N rows][KB] and
  // xq [T rows][G*KB]; one box is KD K blocks of a row tile.
  CUtensorMap tw_map, tx_map;
  {
    const uint64_t wd[3] = {uint64_t(es::kBK), uint64_t(G * N), uint64_t(p.KB)}, wst[2] = {uint64_t(D), 128u};
    const uint64_t xd[3] = {uint64_t(es::kBK), uint64_t(T), uint64_t(G * p.KB)}, xs[2] = {uint64_t(G * D), 128u};
    const uint32_t wb[3] = {uint32_t(es::kBK), uint32_t(bm), uint32_t(p.KD)};
    const uint32_t xb[3] = {uint32_t(es::kBK), uint32_t(mt), uint32_t(p.KD)};
    if (!tensor_map_u8_3d(&tw_map, w_gnd, wd, wst, wb) || !tensor_map_u8_3d(&tx_map, xq, xd, xs, xb))
      return FQ_ERR_CUDA;
  }
  // Schedule: whole tiles when they fill the SMs, else stream-K over one CTA
  // per SM, at least 4 K blocks per CTA (a CTA's fixed cost - tensor-memory
  // set-up, pipeline fill, hand-off - grows with the number of CTAs sharing a
  // tile).  FQ_FORCE_SCHEDULE (tests and studies): dp gives every CTA one
  // whole tile, streamk never rounds to whole tiles, k2 halves each tile;
  // FQ_EINSUM_BM = 64 | 128 fixes the tile rows.
  // stages in flight: about 120 KB per SM (see the W8A8 GEMM's stage cap)
  {
    int ah = (122880 + p.stage / 2) / p.stage;
    if (const char* v = std::getenv("FQ_STAGES_AHEAD")) ah = std::atoi(v);
    p.ahead = ah < 2 ? 2 : (ah > p.S ? p.S : ah);
    // Weight chunks before the wait on the previous kernel: one fewer than the
    // window when it holds three or more.  Copies issued early sit ahead of
    // the activation boxes requested after the wait (GB300, T = 1 / 4 / 16,
    // chained calls: 9.1-9.3 -> 8.9-9.0 us; one chunk measured slower).
    p.pre_w = p.ahead >= 3 ? p.ahead - 1 : 0;
  }
  int64_t by_work = (p.total * p.KD + 3) / 4;
  if (by_work > p.total) by_work = p.total;  // every CTA gets at least one chunk
  int grid = int(by_work < d.sm_count ? (by_work > 0 ? by_work : 1) : d.sm_count);
  const char* f = std::getenv("FQ_FORCE_SCHEDULE");
  if (!f || std::strcmp(f, "streamk")) {
    const int g = whole_tile_grid(tiles, d.sm_count);
    if (g > 0 && g <= grid) grid = g;
  }
  if (f) {
    if (!std::strcmp(f, "dp") && tiles <= es::kMaxGrid) grid = int(tiles);
    // each tile split in two halves (partial sums: the workspace holds two slots per SM)
    if (!std::strcmp(f, "k2") && 2 * tiles <= d.sm_count && p.KB / p.KD >= 2) grid = int(2 * tiles);
  }
  // partial-sum slots exist for sm_count CTAs; only whole-tile CTAs (grid == tiles) may exceed that
  if (grid > d.sm_count && grid != tiles) return FQ_ERR_SHAPE;
  const bool pdl = pdl_enabled();
  cudaError_t e;
  switch (mt) {
    case 16: e = es::launch_es<16>(&tw_map, &tx_map, p, fmt, bm, grid, s, pdl); break;
    case 32: e = es::launch_es<32>(&tw_map, &tx_map, p, fmt, bm, grid, s, pdl); break;
    default: e = es::launch_es<64>(&tw_map, &tx_map, p, fmt, bm, grid, s, pdl); break;
  }
  return cuda_status(e);
}
