// MoE routing kernels: stable sort of (token, slot) pairs by expert id and
// the weighted combine back to token order.
//
// "Reshaping LLM inference dataflow: DeepSeek V4 950", section 3.2: sorting
// tokens by expert id before dispatch keeps each expert's rows contiguous
// (the fix that took the gather from 18% to under 3% of kernel time).
// "DeepSeek-V4 W8A8 performance analysis", section 5: the grouped matmul
// takes group_list = expert_tokens, i.e. the per-expert row counts that the
// offsets below encode; section 1 lists the combine in the layer budget.
#include "fq_common.cuh"

namespace fq {

constexpr int kSortWarps = 8;
constexpr int kMaxExperts = 1024;

// Single-CTA stable counting sort.  The pair list is cut into kSortWarps
// contiguous segments; each warp histograms its segment, the per-expert
// totals are scanned into offsets, each warp's starting cursor per expert is
// offsets[e] plus the counts of the segments before it, and every warp then
// places its segment in order (match_any ranks equal ids inside a 32-pair
// chunk).  The result is the stable order by (expert, pair index).
__global__ void __launch_bounds__(kSortWarps * 32) moe_sort_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                                   int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ perm,
                                                                   int32_t* __restrict__ pair_row,
                                                                   uint32_t* __restrict__ err) {
  extern __shared__ int smem[];
  int* cnt = smem;                       // [kSortWarps][E] counts, then cursors
  int* tot = smem + kSortWarps * E;      // [E + 1] totals, then offsets
  __shared__ int wsum[32];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < kSortWarps * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int seg = (n + kSortWarps - 1) / kSortWarps;
  const int b0 = min(n, warp * seg), b1 = min(n, b0 + seg);
  bool bad = false;
  for (int i = b0 + lane; i < b1; i += 32) {
    const int e = ids[i];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[warp * E + e], 1);
    else
      bad = true;
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(err, DEVERR_BAD_EXPERT_ID);
  __syncthreads();
  // totals and exclusive scan: thread tid owns experts [tid * per, tid * per + per)
  const int per = (E + blockDim.x - 1) / blockDim.x;
  int local = 0;
  for (int k = 0; k < per; ++k) {
    const int e = tid * per + k;
    if (e < E) {
      int s = 0;
      for (int w = 0; w < kSortWarps; ++w) s += cnt[w * E + e];
      tot[e] = s;
      local += s;
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
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += wsum[w];
  int run = wbase + incl - local;  // exclusive prefix of this thread's first expert
  for (int k = 0; k < per; ++k) {
    const int e = tid * per + k;
    if (e < E) {
      const int c = tot[e];
      offsets[e] = run;
      int cur = run;
      for (int w = 0; w < kSortWarps; ++w) {
        const int cw = cnt[w * E + e];
        cnt[w * E + e] = cur;
        cur += cw;
      }
      run += c;
    }
  }
  if (tid == blockDim.x - 1) offsets[E] = run;
  __syncthreads();
  // stable placement, 32 pairs at a time per warp
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = b0; c0 < b1; c0 += 32) {
    const int i = c0 + lane;
    const bool in = i < b1;
    const int e = in ? ids[i] : -1;
    const bool ok = in && e >= 0 && e < E;
    const int key = ok ? e : (E + 1 + lane);  // unique key for lanes that place nothing
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
    if (ok) {
      const int pos = cnt[warp * E + e] + __popc(peers & lt);
      perm[pos] = i;
      if (pair_row) pair_row[i] = pos;
    }
    __syncwarp();
    if (ok && lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

// out[t, :] = bf16_RN( fp32 running sum over slots j = 0..topk-1 of
//                      fp32(w[t, j] * y[pair_row[t*topk + j], :]) ).
// grid = (T, ceil(H / 2048)); each thread owns 8 consecutive columns.
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ pair_row,
                                                          const float* __restrict__ w, int T, int topk, int H8,
                                                          int R, uint4* __restrict__ out, uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (t >= T || c >= H8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < topk; ++j) {
    const int row = pair_row[int64_t(t) * topk + j];
    const float wt = w[int64_t(t) * topk + j];
    if (row < 0 || row >= R) {
      if (c == 0) atomicOr(err, DEVERR_BAD_EXPERT_ID);
      continue;
    }
    const uint4 v = y[int64_t(row) * H8 + c];
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wt, __uint_as_float(q[i] << 16)));
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wt, __uint_as_float(q[i] & 0xFFFF0000u)));
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = uint32_t(f32_to_bf16_bits(acc[2 * i])) | (uint32_t(f32_to_bf16_bits(acc[2 * i + 1])) << 16);
  out[int64_t(t) * H8 + c] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace fq

using namespace fq;

extern "C" __attribute__((visibility("default"))) fq_status moe_sort(const int32_t* topk_ids, int64_t T, int64_t topk, int64_t E, int32_t* offsets,
                              int32_t* perm, int32_t* pair_row, void* ws, size_t ws_bytes, fq_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  if (T < 0 || topk < 0 || E <= 0 || E > kMaxExperts || T * topk > (int64_t(1) << 30)) return FQ_ERR_SHAPE;
  if (!offsets) return FQ_ERR_NULL;
  const int64_t n = T * topk;
  if (n > 0 && (!topk_ids || !perm)) return FQ_ERR_NULL;
  if (!aligned16(offsets) || (n > 0 && (!aligned16(topk_ids) || !aligned16(perm))) ||
      (pair_row && !aligned16(pair_row)))
    return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const size_t smem = (size_t(kSortWarps) * E + E + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(moe_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch(moe_sort_kernel, 1, kSortWarps * 32, smem, reinterpret_cast<cudaStream_t>(stream),
                            pdl_enabled(), topk_ids, int(n), int(E), offsets, perm, pair_row, d.err_word));
}

extern "C" __attribute__((visibility("default"))) fq_status moe_combine(const uint16_t* y_rows, const int32_t* pair_row, const float* topk_w, int64_t T,
                                 int64_t topk, int64_t H, uint16_t* out, fq_stream_t stream) {
  if (T < 0 || topk <= 0 || H < 0 || H % 8 || T > (int64_t(1) << 30) || T * topk > (int64_t(1) << 31) ||
      H > (int64_t(1) << 24))
    return FQ_ERR_SHAPE;
  if (T == 0 || H == 0) return FQ_OK;
  if (!y_rows || !pair_row || !topk_w || !out) return FQ_ERR_NULL;
  if (!aligned16(y_rows) || !aligned16(pair_row) || !aligned16(topk_w) || !aligned16(out)) return FQ_ERR_ALIGN;
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  const int H8 = int(H / 8);
  dim3 grid(unsigned(T), unsigned((H8 + 255) / 256));
  return cuda_status(launch(moe_combine_kernel, grid, 256, 0, reinterpret_cast<cudaStream_t>(stream), pdl_enabled(),
                            reinterpret_cast<const uint4*>(y_rows), pair_row, topk_w, int(T), int(topk), H8,
                            int(T * topk), reinterpret_cast<uint4*>(out), d.err_word));
}
