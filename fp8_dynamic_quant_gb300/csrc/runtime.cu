// Library runtime: status text, CUDA error capture, device checks, the
// per-device error word, tensor-map encoding and workspace sizing.
#include <cstring>
#include <cstdlib>
#include <mutex>

#include "fq_common.cuh"

namespace fq {

// One 32-bit error word per device, in device global memory.  Kernels OR
// flags into it; fq_device_error() reads and clears it.
__device__ uint32_t g_error_word;

static thread_local int t_last_cuda_error = 0;

fq_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FQ_OK;
  t_last_cuda_error = static_cast<int>(e);
  return FQ_ERR_CUDA;
}

static constexpr int kMaxDevices = 64;
static DevInfo g_dev[kMaxDevices];
static std::mutex g_dev_mu;

fq_status device_info(DevInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return FQ_ERR_UNSUPPORTED_DEVICE;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev[dev].id == dev) {
      *info = g_dev[dev];
      return (info->major == 10 && info->minor == 3) ? FQ_OK : FQ_ERR_UNSUPPORTED_DEVICE;
    }
  }
  DevInfo d;
  d.id = dev;
  if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_status(e);
  if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
    return cuda_status(e);
  if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_status(e);
  int optin = 0;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return cuda_status(e);
  d.smem_optin = static_cast<size_t>(optin);
  if (d.major == 10 && d.minor == 3) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess) return cuda_status(e);
    d.err_word = static_cast<uint32_t*>(p);
  }
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    g_dev[dev] = d;
  }
  *info = d;
  return (d.major == 10 && d.minor == 3) ? FQ_OK : FQ_ERR_UNSUPPORTED_DEVICE;
}

int whole_tile_grid(int64_t tiles, int sms) {
  const char* v = std::getenv("FQ_WHOLE_TILES");
  if (v && v[0] == '0') return 0;
  if (tiles <= 0 || sms <= 0) return 0;
  const int64_t per = (tiles + sms - 1) / sms;
  const int64_t g = (tiles + per - 1) / per;
  if (tiles % g != 0) return 0;  // uneven: some tile would still be split
  return g * 4 >= int64_t(sms) * 3 ? int(g) : 0;
}

bool pdl_enabled() {
  static int v = -1;
  if (v < 0) {
    const char* s = std::getenv("FQ_PDL");
    v = (s && s[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {
struct MapEntry {
  const void* ptr;
  uint64_t cols, rows, pitch;
  uint32_t box_cols, box_rows;
  int dev;
  bool valid;
  CUtensorMap map;
};
constexpr int kMapCache = 256;
thread_local MapEntry t_maps[kMapCache];
}  // namespace

// The map is copied into *out: a pointer into the cache would be invalidated
// by the next lookup that hashes to the same slot (a caller holding the weight
// map while encoding the activation map would then launch with the wrong one).
bool tensor_map_u8_2d(CUtensorMap* out, const void* ptr, uint64_t cols, uint64_t rows, uint64_t pitch,
                      uint32_t box_cols, uint32_t box_rows) {
  int dev = 0;
  cudaGetDevice(&dev);
  uint64_t h = reinterpret_cast<uintptr_t>(ptr) >> 4;
  h ^= cols * 0x9E3779B97F4A7C15ull ^ rows * 0xC2B2AE3D27D4EB4Full ^ (uint64_t(box_rows) << 32) ^ box_cols ^
       (uint64_t(dev) << 48) ^ pitch;
  h ^= h >> 29;
  MapEntry& e = t_maps[h % kMapCache];
  if (e.valid && e.ptr == ptr && e.cols == cols && e.rows == rows && e.pitch == pitch &&
      e.box_cols == box_cols && e.box_rows == box_rows && e.dev == dev) {
    *out = e.map;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    e.valid = false;
    return false;
  }
  e.ptr = ptr;
  e.cols = cols;
  e.rows = rows;
  e.pitch = pitch;
  e.box_cols = box_cols;
  e.box_rows = box_rows;
  e.dev = dev;
  e.valid = true;
  *out = e.map;
  return true;
}

namespace {
struct Map3Entry {
  const void* ptr;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  int dev;
  bool valid;
  CUtensorMap map;
};
constexpr int kMap3Cache = 128;
thread_local Map3Entry t_maps3[kMap3Cache];
}  // namespace

bool tensor_map_u8_3d(CUtensorMap* out, const void* ptr, const uint64_t dims[3], const uint64_t strides[2],
                      const uint32_t box[3]) {
  int dev = 0;
  cudaGetDevice(&dev);
  uint64_t h = reinterpret_cast<uintptr_t>(ptr) >> 4;
  for (int i = 0; i < 3; ++i) h = (h ^ dims[i]) * 0x9E3779B97F4A7C15ull ^ (uint64_t(box[i]) << (16 * i));
  h ^= strides[0] * 0xC2B2AE3D27D4EB4Full ^ strides[1] ^ (uint64_t(dev) << 48);
  h ^= h >> 29;
  Map3Entry& e = t_maps3[h % kMap3Cache];
  if (e.valid && e.ptr == ptr && e.dev == dev && e.dims[0] == dims[0] && e.dims[1] == dims[1] &&
      e.dims[2] == dims[2] && e.strides[0] == strides[0] && e.strides[1] == strides[1] && e.box[0] == box[0] &&
      e.box[1] == box[1] && e.box[2] == box[2]) {
    *out = e.map;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), d, st, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    e.valid = false;
    return false;
  }
  e.ptr = ptr;
  for (int i = 0; i < 3; ++i) {
    e.dims[i] = dims[i];
    e.box[i] = box[i];
  }
  e.strides[0] = strides[0];
  e.strides[1] = strides[1];
  e.dev = dev;
  e.valid = true;
  *out = e.map;
  return true;
}

// One warp: lane 0 waits on an mbarrier that only it can complete.  The
// wait is the library's bounded wait; when it gives up, the timeout flag is
// recorded exactly as the pipelined kernels record it.
__global__ void selftest_wait_kernel(uint64_t budget_ns, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    if (!mbar_wait_ns(&bar, 0, budget_ns)) atomicOr(&g_error_word, DEVERR_TIMEOUT);
  }
  __syncwarp();
}

}  // namespace fq

using namespace fq;

extern "C" __attribute__((visibility("default"))) fq_status fq_selftest_wait_timeout(uint64_t budget_ns, int arrive,
                                                                                     fq_stream_t stream) {
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  if (budget_ns < 1000ull) budget_ns = 1000ull;
  if (budget_ns > 1000000000ull) budget_ns = 1000000000ull;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_ns, arrive);
  return cuda_status(cudaGetLastError());
}

extern "C" __attribute__((visibility("default"))) const char* fq_status_string(int s) {
  switch (s) {
    case FQ_OK: return "ok";
    case FQ_ERR_NULL: return "a required pointer is NULL";
    case FQ_ERR_SHAPE: return "invalid shape (negative, too large, or breaks a divisibility rule)";
    case FQ_ERR_ALIGN: return "pointer is not 16-byte aligned";
    case FQ_ERR_WORKSPACE: return "workspace missing or too small";
    case FQ_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
    case FQ_ERR_CUDA: return "CUDA call failed (see fq_last_cuda_error)";
    case FQ_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case FQ_ERR_DEVICE_INPUT: return "device input broke the contract (e.g. expert id out of range)";
    case FQ_ERR_ARG: return "invalid argument value (unknown enum, bad eps, overlapping buffers)";
    default: return "unknown status";
  }
}

extern "C" __attribute__((visibility("default"))) int fq_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" __attribute__((visibility("default"))) fq_status fq_device_error(fq_stream_t stream, uint32_t* detail) {
  DevInfo d;
  fq_status st = device_info(&d);
  if (st != FQ_OK) return st;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t w = 0, zero = 0;
  if ((e = cudaMemcpy(&w, d.err_word, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_status(e);
  if ((e = cudaMemcpy(d.err_word, &zero, 4, cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_status(e);
  if (detail) *detail = w;
  if (w & DEVERR_TIMEOUT) return FQ_ERR_DEVICE_TIMEOUT;
  if (w) return FQ_ERR_DEVICE_INPUT;
  return FQ_OK;
}

extern "C" __attribute__((visibility("default"))) fq_status fq_check_device_error(fq_stream_t stream) {
  return fq_device_error(stream, nullptr);
}

extern "C" __attribute__((visibility("default"))) size_t fq_workspace_bytes(int op, int64_t a, int64_t b, int64_t c, int64_t d) {
  if (a < 0 || b < 0 || c < 0 || d < 0) return 0;
  switch (op) {
    case FQ_OP_W8A8_LINEAR: return ws_w8a8_linear(a, b, c);
    case FQ_OP_W8A8_QUANT_LINEAR: return ws_w8a8_quant_linear(a, b, c);
    case FQ_OP_FP8_GROUP_EINSUM: return ws_fp8_group_einsum(a, b, c, d);
    case FQ_OP_MOE_SORT: return 256;
    case FQ_OP_W8A8_GROUPED_LINEAR: return ws_w8a8_grouped_linear(a, b, c, d);
    case FQ_OP_MXFP8_LINEAR: return ws_mxfp8_linear(a, b, c);
    default: return 0;
  }
}
