// host_util.cu -- tensor-map encoding (through the driver entry point, so the
// library needs no link-time libcuda) and the device error word.
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/bpt.h"

#include "internal.h"
#include "ptx.cuh"

namespace bpt {

__device__ unsigned int g_err[4];

// The per-device caches below are atomics: host threads may call the library
// concurrently, and each would store the same value.
unsigned int* device_error_word() {
  static std::atomic<unsigned int*> addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned int* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err) != cudaSuccess) return nullptr;
    a = reinterpret_cast<unsigned int*>(p);
    addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

struct ProfRec {
  cudaEvent_t a = nullptr, b = nullptr;
  int kind = 0;
  double flops = 0, bytes = 0;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};  // read without the lock on every launch
std::vector<ProfRec> g_prof;
size_t g_prof_used = 0;

}  // namespace

ProfScope::ProfScope(int kind, double flops, double bytes, cudaStream_t s) : slot(-1), st(s) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  if (g_prof_used == g_prof.size()) {
    ProfRec r;
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
    g_prof.push_back(r);
  }
  slot = (int)g_prof_used++;
  g_prof[slot].kind = kind;
  g_prof[slot].flops = flops;
  g_prof[slot].bytes = bytes;
  cudaEventRecord(g_prof[slot].a, st);
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEventRecord(g_prof[slot].b, st);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cached.store(fn, std::memory_order_release);
  }
  return fn;
}

CUtensorMapSwizzle swz(int bytes) {
  switch (bytes) {
    case 32: return CU_TENSOR_MAP_SWIZZLE_32B;
    case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
    case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
    default: return CU_TENSOR_MAP_SWIZZLE_NONE;
  }
}

}  // namespace

int make_map_2d(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                uint32_t box_cols, uint32_t box_rows, int swizzle_bytes, int elem_bytes) {
  auto fn = encode_fn();
  if (!fn || !ptr) return 1;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || ((ld * elem_bytes) & 15)) return 1;
  if (box_rows > 256 || box_cols > 256) return 1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz(swizzle_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 1;
}

// 3-D map over a packed [b, s, ld] bf16 buffer: x = column, y = row in the
// sequence, z = sequence.  Rows past s read as zeros within each sequence.
// box = {chunk width, 128, 1}: 64 columns with 128-byte swizzle when d is a
// multiple of 64, else 16 columns with 32-byte swizzle.
int make_attn_map(CUtensorMap* map, const void* qkv, int b, int s, int64_t ld, int d) {
  auto fn = encode_fn();
  if (!fn || !qkv) return 1;
  if ((reinterpret_cast<uintptr_t>(qkv) & 15) || ((ld * 2) & 15)) return 1;
  const int cw = (d % 64 == 0) ? 64 : 16;
  cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)s, (cuuint64_t)b};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * (cuuint64_t)s};
  cuuint32_t box[3] = {(cuuint32_t)cw, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, cw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 1;
}

// Watchdog self-test.  One thread waits, through the same bounded_wait every
// kernel of the library uses, on an mbarrier that nothing ever arrives at.
// The wait gives up after BPT_WAIT_CYCLES SM cycles, records `site` in the
// error word and returns; the kernel then leaves normally, so the context
// stays usable.  Nothing is faulted: the stall is a barrier nobody signals.
__global__ void watchdog_selftest_kernel(unsigned int* err, int site) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  bounded_wait(&bar, 0, &abort_flag, site, err);
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
}

// [p, p + bytes) inside one device allocation of the current device: the
// runtime classifies the pointer (device or managed memory, on this device)
// and the driver gives the allocation holding it (its base and size), taken
// through the driver entry point like the tensor-map encoder.
typedef CUresult (*PfnMemGetAddressRange)(CUdeviceptr*, size_t*, CUdeviceptr);

int check_device_range(const void* p, size_t bytes) {
  if (!p) return 1;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // the query's error is not the caller's
    return 1;
  }
  if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != dev) return 1;
  static std::atomic<PfnMemGetAddressRange> cached{nullptr};
  PfnMemGetAddressRange fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return 1;
    fn = reinterpret_cast<PfnMemGetAddressRange>(f);
    cached.store(fn, std::memory_order_release);
  }
  CUdeviceptr base = 0;
  size_t size = 0;
  if (fn(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return 1;
  const uint64_t lo = reinterpret_cast<uint64_t>(p);
  return (lo >= base && bytes <= size && lo - base <= size - bytes) ? 0 : 1;
}

// Reads and clears the error word (synchronising the stream first).
int read_device_error(cudaStream_t st, unsigned int out[4]) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    out[0] = 3;
    out[1] = (unsigned)e;
    return 3;
  }
  unsigned int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(out, g_err, sizeof(unsigned int) * 4) != cudaSuccess) return 3;
  if (cudaMemcpyToSymbol(g_err, zero, sizeof(zero)) != cudaSuccess) return 3;
  return 0;
}

}  // namespace bpt

extern "C" {

int bpt_check_device_range(const void* ptr, size_t bytes) {
  return bpt::check_device_range(ptr, bytes) ? BPT_EINVAL : BPT_OK;
}

int bpt_watchdog_selftest(void* stream) {
  unsigned int* err = bpt::device_error_word();
  if (!err) return BPT_ECUDA;
  bpt::watchdog_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      err, BPT_WATCHDOG_SELFTEST_SITE);
  return cudaGetLastError() == cudaSuccess ? BPT_OK : BPT_ECUDA;
}

int bpt_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(bpt::g_prof_mu);
  bpt::g_prof_on = on != 0;
  bpt::g_prof_used = 0;
  return BPT_OK;
}

int bpt_profile_list(int max, int* kind, double* flops, double* bytes, double* ms) {
  if (max < 0 || (max > 0 && (!kind || !flops || !bytes || !ms))) return -BPT_EINVAL;
  std::lock_guard<std::mutex> lk(bpt::g_prof_mu);
  const int n = (int)std::min<size_t>((size_t)max, bpt::g_prof_used);
  for (int i = 0; i < n; ++i) {
    auto& r = bpt::g_prof[i];
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -BPT_ECUDA;
    float t = 0;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -BPT_ECUDA;
    kind[i] = r.kind;
    flops[i] = r.flops;
    bytes[i] = r.bytes;
    ms[i] = t;
  }
  return n;
}

int bpt_profile_collect(int nkinds, double* ms, double* flops, double* bytes, int* launches) {
  if (nkinds < 1 || !ms || !flops || !bytes || !launches) return BPT_EINVAL;
  std::lock_guard<std::mutex> lk(bpt::g_prof_mu);
  for (int k = 0; k < nkinds; ++k) {
    ms[k] = flops[k] = bytes[k] = 0;
    launches[k] = 0;
  }
  for (size_t i = 0; i < bpt::g_prof_used; ++i) {
    auto& r = bpt::g_prof[i];
    if (cudaEventSynchronize(r.b) != cudaSuccess) return BPT_ECUDA;
    float t = 0;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return BPT_ECUDA;
    if (r.kind < nkinds) {
      ms[r.kind] += t;
      flops[r.kind] += r.flops;
      bytes[r.kind] += r.bytes;
      launches[r.kind] += 1;
    }
  }
  bpt::g_prof_used = 0;
  return BPT_OK;
}

}  // extern "C"
