// Shared device/host helpers of libssd (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "ssd.h"

namespace ssd {

// ---------------------------------------------------------------- host side
extern std::atomic<uint64_t> g_launches;

inline void count_launch(uint64_t n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

// measurement hook: events recorded around chosen kernels (ssd_profile_kernel)
constexpr int kProfileSlots = 16;
struct ProfileHook {
  std::atomic<int> on[kProfileSlots];
  cudaEvent_t start[kProfileSlots];
  cudaEvent_t end[kProfileSlots];
};
extern ProfileHook g_profile;

inline void record_hook_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else cudaEventRecord(ev, s);
}

// RAII bracket: records the kernel's start event on construction and its end
// event on destruction while kernel `id` is being profiled
struct KernelTimer {
  cudaStream_t s;
  int id;
  bool on;
  KernelTimer(int kid, cudaStream_t st) : s(st), id(kid), on(g_profile.on[kid].load(std::memory_order_relaxed) != 0) {
    if (on) record_hook_event(g_profile.start[id], s);
  }
  ~KernelTimer() {
    if (on) record_hook_event(g_profile.end[id], s);
  }
};

// Launch with programmatic dependent launch allowed: the kernel may start while
// the previous kernel of the stream finishes; it must execute
// `griddepcontrol.wait` before reading that kernel's outputs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Kernel attributes, occupancy figures and the static scratch address are per device:
// host-side caches of them are arrays indexed by the current device.
constexpr int kMaxDevices = 64;

// the current device as an index into such a cache, or -1
inline int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every workspace starts with this header. err is the device error word.
struct WsHeader {
  int32_t err;        // SSD_OK or the first device-side error recorded
  int32_t where;      // diagnostic: which wait / check recorded it
  int32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ---------------------------------------------------------------- device side
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16, round to nearest even (finite inputs)
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ void record_error(WsHeader* h, int code, int where) {
  if (h != nullptr && atomicCAS(&h->err, 0, code) == 0) h->where = where;
}

// ---------------------------------------------------------------- checked builds
// A build with -DSSD_CHECKS=1 (libssd_checked.so) tests every guarded index against the
// extent it must stay within before the access; a failed test records SSD_ERR_DEVICE with
// `where` in the call's workspace header (when the call has one) and in the check word of
// the translation unit (read with ssd_read_check_error), and the access is skipped. In the
// normal build the tests compile away.
#ifndef SSD_CHECKS
#define SSD_CHECKS 0
#endif
#if SSD_CHECKS
static __device__ WsHeader g_check_word;
#endif

__device__ __forceinline__ bool in_range(long long i, long long n, WsHeader* hdr, int where) {
#if SSD_CHECKS
  if (i >= 0 && i < n) return true;
  record_error(hdr, SSD_ERR_DEVICE, where);
  record_error(&g_check_word, SSD_ERR_DEVICE, where);
  return false;
#else
  (void)i; (void)n; (void)hdr; (void)where;
  return true;
#endif
}

// host: every translation unit of a checked build registers a reader of its check word
typedef int (*CheckWordReader)(cudaStream_t s, int32_t* out);
void register_check_word(CheckWordReader f);
#if SSD_CHECKS
static int read_check_word(cudaStream_t s, int32_t* out) {
  void* a = nullptr;
  if (cudaGetSymbolAddress(&a, g_check_word) != cudaSuccess) return SSD_ERR_CUDA;
  int32_t w[2] = {0, 0};
  if (cudaMemcpyAsync(w, a, sizeof w, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  if (w[0] != 0) {
    const int32_t z[2] = {0, 0};
    if (cudaMemcpyAsync(a, z, sizeof z, cudaMemcpyHostToDevice, s) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  }
  *out = w[0];
  return SSD_OK;
}
namespace {
struct CheckWordRegistration {
  CheckWordRegistration() { register_check_word(&read_check_word); }
};
static CheckWordRegistration g_check_word_registration;
}  // namespace
#endif

// One probe of an mbarrier phase (shared memory of this CTA): true once the phase of the
// given parity has completed.
__device__ __forceinline__ bool mbar_probe(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity)
      : "memory");
  return ok != 0;
}

// The library's bounded wait: after `limit` clocks without the phase completing it sets
// *failed (so that the CTA's other waits return at once), records SSD_ERR_TIMEOUT with
// `where` in the workspace header and returns false; it never traps.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* failed, WsHeader* hdr,
                                                  int where, unsigned long long limit) {
  if (mbar_probe(bar, parity)) return true;      // the common case: one probe, no bookkeeping
  if (*failed) return false;
  const unsigned long long t0 = clock64();
  while (!mbar_probe(bar, parity)) {
    if (*failed) return false;
    if (clock64() - t0 > limit) {
      *failed = 1;
      record_error(hdr, SSD_ERR_TIMEOUT, where);
      return false;
    }
  }
  return true;
}

constexpr float kLog2e = 1.4426950408889634f;

// 2^x, hardware approximation (MUFU), flush-to-zero
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace ssd
