// attn_bwd_noalloc.cu -- bpt_attention_bwd_noalloc: the attention backward
// with its scratch (the per-row dO . O sums and -LSE * log2(e)) in a fixed
// array compiled into the library, for callers that cannot allocate device memory when they
// call us.
//
// Who cannot allocate: code that must run with a device-memory plan fixed
// ahead of time -- an inference or training engine's plugin whose enqueue
// step may not call cudaMalloc, a caller that cannot afford cudaMalloc /
// cudaFree (which may synchronise the device) on its hot path, or a process
// whose memory is carved up by another allocator that owns every byte.  Such
// a caller passes only its inputs and outputs; the scratch lives here.
//
// The array costs BPT_NOALLOC_SCRATCH_BYTES of device memory on every GPU
// that loads this part of the library, for the life of the process.  Every
// call shares it: two calls that overlap on the GPU (different streams, or
// different host threads on one device) race on it and produce wrong results,
// so serialise them.  A call fully overwrites the part of the array it uses,
// so nothing has to start at zero.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bpt.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_attn_bwd_scratch[BPT_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  Host code may
// not use the symbol itself as a pointer (on the host it names a host-side
// stand-in), so the address is looked up once per device, with that device
// current, and cached.
void* scratch_on_current_device(int* status) {
  static std::atomic<void*> addr[64];  // host threads may race here; all store the same value
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = BPT_ECUDA;
    return nullptr;
  }
  void* p = addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_attn_bwd_scratch) != cudaSuccess || !p) {
      *status = BPT_ECUDA;
      return nullptr;
    }
    addr[dev].store(p, std::memory_order_release);
  }
  *status = BPT_OK;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int bpt_attention_bwd_noalloc(const bpt_config* cfg, const void* qkv, const void* o,
                                         const void* lse, const void* dout, void* dqkv, void* stream) {
  if (!cfg || !qkv || !o || !lse || !dout || !dqkv) return BPT_EINVAL;
  if (!aligned16(qkv) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) || !aligned16(dqkv))
    return BPT_EINVAL;
  // the same validation and geometry as bpt_attention_bwd
  const size_t need = bpt_attention_bwd_workspace_bytes(cfg);
  if (need == 0) {
    // invalid or unsupported: let the regular entry point classify it without
    // touching any memory (a null workspace fails its checks before launch)
    return bpt_attention_bwd(cfg, qkv, o, lse, dout, dqkv, nullptr, 0, stream);
  }
  if (need > (size_t)BPT_NOALLOC_SCRATCH_BYTES) return BPT_ENOSPC;
  int st = BPT_OK;
  void* scratch = scratch_on_current_device(&st);
  if (!scratch) return st;
  return bpt::attention_bwd_call(cfg, qkv, o, lse, dout, dqkv, scratch, (size_t)BPT_NOALLOC_SCRATCH_BYTES, stream,
                                1);
}
