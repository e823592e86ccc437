// Shared device helpers and host-side plumbing for the fq library (sm_103a).
//
// Everything here is infrastructure: inline-PTX wrappers for mbarriers, TMA
// (cp.async.bulk.tensor), programmatic dependent launch, and the host
// validation / launch helpers used by every entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>
#include <cstddef>

#include "../../include/fq.h"

namespace fq {

// ------------------------------------------------------------ device error word
// Bit flags OR-ed into the per-device error word.
enum : uint32_t {
  DEVERR_TIMEOUT = 1u,        // a bounded mbarrier wait gave up
  DEVERR_BAD_EXPERT_ID = 2u,  // moe_sort met an id outside [0, E)
};

// Wall-clock bound of every device-side wait (nanoseconds, %globaltimer).
constexpr uint64_t kWaitNs = 200ull * 1000ull * 1000ull;

// ------------------------------------------------------------ small device helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Store to global memory through the global state space (no aliasing with
// shared memory for the compiler to assume).
__device__ __forceinline__ void st_global_u16(uint16_t* p, uint16_t v) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on phase `parity`; false if it did not complete within
// `budget_ns` of wall-clock time.
__device__ __forceinline__ bool mbar_wait_ns(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > budget_ns) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_ns(bar, parity, kWaitNs);
}
// Wait for tensor-core issue loops: one try_wait inline; the CTA's abort flag
// and the bounded polling loop only once the phase is found incomplete, out of
// line.  Inlined, the loop and its timer reads, or a shared-memory flag read
// per wait, slowed an MMA issue loop by ~60-100 ns per wait on GB300 even when
// the phase had already completed.  (Loops whose waits usually block keep the
// inline mbar_wait: a call there costs more than it saves.)
static __device__ __noinline__ bool mbar_wait_slow_or_abort(uint64_t* bar, uint32_t parity,
                                                            volatile int* abort_flag) {
  return !*abort_flag && mbar_wait(bar, parity);
}
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow_or_abort(bar, parity, abort_flag);
}
// The same order with the polling loop inline, for loops whose waits often block.
__device__ __forceinline__ bool mbar_wait_try_first(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || (!*abort_flag && mbar_wait(bar, parity));
}

// ------------------------------------------------------------ TMA (tensor copies)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// 2-D tiled load global -> shared, completion counted on `bar` in bytes.
// x is the innermost coordinate (in elements); for 8-bit data it must be a
// multiple of 16 (every caller passes multiples of 128).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// 3-D tiled load global -> shared (coordinates innermost first), completion
// counted on `bar` in bytes.  x must be a multiple of 16 for 8-bit data.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
// 1-D bulk copy global -> shared (the TMA engine), completion counted on
// `bar` in bytes.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------ programmatic dependent launch
// Wait until the preceding kernel in the stream has finished and its writes
// are visible (no-op when the launch was not programmatic).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to start launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Split-K arrival: acq_rel atomic add at GPU scope.  The release half
// publishes this CTA's partial sums (ordered before it by a CTA barrier);
// the acquire half lets the last arriving CTA read everyone else's.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of all CTAs in the cluster; release/acquire orders shared-memory
// (incl. distributed shared memory) accesses across the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split form: arrive early, wait later (the wait acquires what arrivals released).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------ tcgen05 (5th-gen tensor cores, TMEM)
// One warp allocates `ncols` (power of two >= 32) tensor-memory columns; the
// base address (lane 0, first column) is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// One lane of a converged warp (elect.sync over the full mask): the issuing
// lane of warp-wide tensor-core loops.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t.reg .b32 R;\n\telect.sync R|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}\n"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row atoms of 1024 bytes (stride
// byte offset), the leading byte offset unused.  `saddr` is the shared
// address of the first row's first 16-byte chunk for this K step; advancing
// along K inside the 128-byte row is a plain address offset.
__device__ __forceinline__ uint64_t umma_desc_k_sw128(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;            // leading byte offset (16 B, ignored for this layout)
  d |= uint64_t(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;            // descriptor version
  d |= uint64_t(2) << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16 with f16 A and B (both K-major) and an
// fp32 accumulator, tile M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Warp-wide store of 32 consecutive 32-bit columns: lane i of the warp
// writes row (taddr.lane + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// Warp-wide loads of 16 / 32 consecutive 32-bit columns (lane i: row taddr.lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// ------------------------------------------------------------ host side
// Device properties of the current device, cached per device id.
struct DevInfo {
  int id = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
  size_t smem_optin = 0;
  uint32_t* err_word = nullptr;  // device address of this device's error word
};
// Fills *info for the current device; FQ_ERR_UNSUPPORTED_DEVICE unless sm_103.
fq_status device_info(DevInfo* info);

// Records a CUDA error for fq_last_cuda_error() and maps it to a status.
fq_status cuda_status(cudaError_t e);

// Encodes a 2-D 8-bit tensor map (inner dimension `cols` bytes, `rows` rows,
// row pitch `pitch` bytes) with a box of box_cols x box_rows and 128-byte
// swizzle, written to *out; encodings are cached per thread by (ptr, sizes).
// Returns false on failure.
bool tensor_map_u8_2d(CUtensorMap* out, const void* ptr, uint64_t cols, uint64_t rows, uint64_t pitch,
                      uint32_t box_cols, uint32_t box_rows);

// Encodes a 3-D 8-bit tensor map: dims[0] the innermost extent in bytes,
// strides[0] / strides[1] the byte strides of dimensions 1 and 2 (any order of
// magnitude: a K-block axis of stride 128 under a row axis of stride D lets
// one box fetch several K blocks of a row tile, landing as consecutive
// 128-byte-swizzled K-major sub-tiles); box[i] elements per dimension.
// Cached per thread like the 2-D maps.  Returns false on failure.
bool tensor_map_u8_3d(CUtensorMap* out, const void* ptr, const uint64_t dims[3], const uint64_t strides[2],
                      const uint32_t box[3]);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with (optional) programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launch with a 1-D thread-block cluster of `cluster` CTAs (and optional PDL).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           bool pdl, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Whether launches may use programmatic dependent launch (env FQ_PDL=0 turns it off).
bool pdl_enabled();

// ---------------------------------------------------------------- per-token INT8 quant math
// (shared by the quant kernels and the GEMM that quantizes its own activations)

// q = clamp(rint(x / s), -127, 127) with x / s the IEEE fp32 quotient, ties
// to even.  The quotient is first estimated as x * RN(1/s) (within 2.3e-5 of
// the IEEE quotient for |x / s| <= 127); only when that estimate lies within
// 2^-14 of a half-integer, where the two could round differently, is the
// exact __fdiv_rn taken.  s == 0 only for an all-zero row (q = 0).  When
// RN(1/s) is not finite (s below ~2.9e-39) every element takes the exact path.
__device__ __forceinline__ int quant_i8(float x, float s, float inv_s) {
  if (s == 0.0f) return 0;
  const float y = __fmul_rn(x, inv_s);
  float r = rintf(y);
  const float d = fabsf(y - r);
  if (!(fabsf(d - 0.5f) >= (1.0f / 16384.0f))) r = rintf(__fdiv_rn(x, s));  // also catches NaN from inf
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return static_cast<int>(r);
}

__device__ __forceinline__ uint32_t pack4_i8(int a, int b, int c, int d) {
  return (uint32_t(a) & 0xFFu) | ((uint32_t(b) & 0xFFu) << 8) | ((uint32_t(c) & 0xFFu) << 16) |
         ((uint32_t(d) & 0xFFu) << 24);
}

// 8 bf16 values in a uint4 -> floats.
__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float absmax8(const float f[8]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// Packed fp32 pairs (Blackwell's f32x2 multiply, add and subtract): each half
// is the IEEE round-to-nearest-even result, subnormals kept, the same value
// as the scalar __fmul_rn / __fadd_rn / __fsub_rn; one instruction for two.
__device__ __forceinline__ float2 f2_op_mul(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_op_add(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_op_sub(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// max(a, |b|, |c|) propagating NaN (three-input PTX max.NaN).
__device__ __forceinline__ float max_abs2_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

// Eight codes with the rule above.  Fast path: y = x * RN(1/s); adding
// 1.5 * 2^23 rounds y to an integer (ties to even) held in the low bits, so
// the low byte is the two's-complement code, and subtracting it back gives
// rint(y).  The largest |y - rint(y)| and |y| of the eight (NaN propagating)
// decide for all eight at once: if any lies within 2^-14 of a half-integer,
// rounds beyond +-127 (the clamp) or is not a number (s == 0, RN(1/s) not
// finite, a NaN or infinite input), all eight take the exact per-element
// path.  The fast path works on pairs (f32x2) and three-input maxima.
// Identical codes, a fraction of the per-element path's instructions (the
// many-rows kernel is issue-bound on GB300).
__device__ __forceinline__ uint2 quant8_i8(const float f[8], float s, float inv) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float2 inv2 = make_float2(inv, inv), mg = make_float2(kMagic, kMagic);
  uint32_t t[8];
  float dmax = 0.0f, ymax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 y = f2_op_mul(make_float2(f[2 * i], f[2 * i + 1]), inv2);
    const float2 tm = f2_op_add(y, mg);
    const float2 d = f2_op_sub(y, f2_op_sub(tm, mg));
    dmax = max_abs2_nan(dmax, d.x, d.y);
    ymax = max_abs2_nan(ymax, y.x, y.y);
    t[2 * i] = __float_as_uint(tm.x);
    t[2 * i + 1] = __float_as_uint(tm.y);
  }
  uint2 o;
  if (dmax < 0.5f - 1.0f / 16384.0f && ymax < 127.5f) {
    o.x = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    o.y = __byte_perm(__byte_perm(t[4], t[5], 0x0040), __byte_perm(t[6], t[7], 0x0040), 0x5410);
  } else {
    o.x = pack4_i8(quant_i8(f[0], s, inv), quant_i8(f[1], s, inv), quant_i8(f[2], s, inv), quant_i8(f[3], s, inv));
    o.y = pack4_i8(quant_i8(f[4], s, inv), quant_i8(f[5], s, inv), quant_i8(f[6], s, inv), quant_i8(f[7], s, inv));
  }
  return o;
}

// max |x| of 8 bf16 values as fp32, on packed pairs: sign bits cleared, then
// bf16x2 max (a NaN is ignored, as fmaxf ignores it); the same value as
// absmax8 of the unpacked floats.
__device__ __forceinline__ float absmax8_bf16(const uint4& v) {
  const uint32_t w0 = v.x & 0x7FFF7FFFu, w1 = v.y & 0x7FFF7FFFu, w2 = v.z & 0x7FFF7FFFu, w3 = v.w & 0x7FFF7FFFu;
  const __nv_bfloat162 m01 = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w0),
                                     *reinterpret_cast<const __nv_bfloat162*>(&w1));
  const __nv_bfloat162 m23 = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w2),
                                     *reinterpret_cast<const __nv_bfloat162*>(&w3));
  const __nv_bfloat162 m = __hmax2(m01, m23);
  return fmaxf(__low2float(m), __high2float(m));
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace fq

namespace fq {
// Every workspace starts with the same fixed block of per-tile arrival
// counters (kMaxTiles words), so workspaces can be shared by different ops
// and shapes: scratch of one call never lands on the counters of another.
constexpr int64_t kMaxTiles = 65536;
constexpr size_t kCounterBytes = size_t(kMaxTiles) * 4;
// Workspace sizes of each op (bytes), for the current device.
size_t ws_w8a8_linear(int64_t M, int64_t K, int64_t N);
size_t ws_w8a8_quant_linear(int64_t M, int64_t K, int64_t N);
size_t ws_fp8_group_einsum(int64_t T, int64_t D, int64_t N, int64_t G);
size_t ws_w8a8_grouped_linear(int64_t R, int64_t K, int64_t N, int64_t E);
// Per-token INT8 quant; trigger: let the next kernel launch before this one
// finishes (only where the output is activations).
fq_status quant_int8_launch(const uint16_t* x, int64_t M, int64_t K, int8_t* xq, float* sx, fq_stream_t stream,
                            bool trigger);
size_t ws_mxfp8_linear(int64_t M, int64_t K, int64_t N);
constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// Stream-K grid that hands every CTA whole tiles when that still fills at
// least 3/4 of the SMs: with ceil(tiles / sms) tiles a CTA, the CTA count is
// ceil(tiles / that), and a tile count that it divides leaves no tile split
// between CTAs - no partial sums, no hand-off at the end.  Returns 0 when the
// whole-tile grid would leave more than a quarter of the SMs idle.  Env
// FQ_WHOLE_TILES=0 turns it off (studies).
int whole_tile_grid(int64_t tiles, int sms);
}  // namespace fq
