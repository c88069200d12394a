// Library-wide entry points: status strings, version, launch counter, the device
// error word and the self-test of the bounded waits.
#include "ssd_common.cuh"

extern "C" const char* ssd_status_string(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported shape or type";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSD_ERR_TIMEOUT: return "device-side wait timed out";
    case SSD_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
  }
}

extern "C" int ssd_version(void) { return 100; }

namespace ssd {
static CheckWordReader g_check_readers[32];
static int g_check_reader_count = 0;
void register_check_word(CheckWordReader f) {
  if (g_check_reader_count < 32) g_check_readers[g_check_reader_count++] = f;
}
}  // namespace ssd

extern "C" int ssd_checked_build(void) { return SSD_CHECKS ? 1 : 0; }

extern "C" int ssd_read_check_error(void* stream, int32_t* out) {
  if (out == nullptr) return SSD_ERR_INVALID;
  int32_t first = SSD_OK;
  for (int i = 0; i < ssd::g_check_reader_count; ++i) {
    int32_t w = SSD_OK;
    const int rc = ssd::g_check_readers[i](static_cast<cudaStream_t>(stream), &w);
    if (rc != SSD_OK) return rc;
    if (first == SSD_OK) first = w;
  }
  *out = first;
  return SSD_OK;
}

namespace ssd {
ProfileHook g_profile;
}

extern "C" int ssd_profile_kernel(int kernel_id, void* start_event, void* end_event) {
  using ssd::g_profile;
  if (kernel_id < SSD_KERNEL_NONE || kernel_id > SSD_KERNEL_HEAD_COMBINE) return SSD_ERR_INVALID;
  if (kernel_id == SSD_KERNEL_NONE) {
    for (int i = 0; i < ssd::kProfileSlots; ++i) g_profile.on[i].store(0);
    return SSD_OK;
  }
  if (start_event == nullptr || end_event == nullptr) return SSD_ERR_INVALID;
  g_profile.on[kernel_id].store(0);
  g_profile.start[kernel_id] = static_cast<cudaEvent_t>(start_event);
  g_profile.end[kernel_id] = static_cast<cudaEvent_t>(end_event);
  g_profile.on[kernel_id].store(1);
  return SSD_OK;
}

extern "C" uint64_t ssd_launch_count(void) { return ssd::g_launches.load(std::memory_order_relaxed); }

extern "C" int ssd_read_device_error(void* ws, void* stream, int32_t* out) {
  if (ws == nullptr || out == nullptr) return SSD_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host[2] = {0, 0};
  if (cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  const int32_t zero[2] = {0, 0};
  if (host[0] != 0) {
    if (cudaMemcpyAsync(ws, zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess) return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  }
  *out = host[0];
  return SSD_OK;
}

namespace ssd {
// one CTA: an mbarrier that is arrived on (arrive != 0) or never, waited on with the
// library's bounded wait
__global__ void k_selftest_wait(WsHeader* hdr, int arrive, unsigned long long limit) {
  __shared__ uint64_t bar;
  __shared__ int failed;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&bar)))
                 : "memory");
    failed = 0;
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0)
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&bar)))
                 : "memory");
  mbar_wait_bounded(&bar, 0, &failed, hdr, 99, limit);
  __syncthreads();
}
}  // namespace ssd

extern "C" int ssd_selftest_wait(void* ws, int arrive, uint64_t limit_clocks, void* stream) {
  if (limit_clocks < 1 || limit_clocks > (1ull << 32)) return SSD_ERR_INVALID;
  if (ws == nullptr || !ssd::aligned(ws, 256)) return SSD_ERR_WORKSPACE;
  ssd::k_selftest_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<ssd::WsHeader*>(ws), arrive,
                                                                         static_cast<unsigned long long>(limit_clocks));
  ssd::count_launch();
  return ssd::check_launch();
}

// ------------------------------------------------------------------ read-bandwidth probe
namespace ssd {
// Every thread keeps 8 independent 16-byte loads in flight per pass of a grid-stride
// loop over the buffer and folds them into an XOR; the fold is stored only if it equals
// a value the caller passes (never, for a buffer that does not hold it), so the loads
// cannot be dropped and nothing but `sink` is ever written.
__global__ void __launch_bounds__(256) k_read_probe(const uint4* __restrict__ buf, size_t nvec, uint4* sink,
                                                    uint32_t magic) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  for (; i + 7 * stride < nvec; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldg(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc.x ^= v[u].x;
      acc.y ^= v[u].y;
      acc.z ^= v[u].z;
      acc.w ^= v[u].w;
    }
  }
  for (; i < nvec; i += stride) {
    const uint4 v = __ldg(buf + i);
    acc.x ^= v.x;
    acc.y ^= v.y;
    acc.z ^= v.z;
    acc.w ^= v.w;
  }
  if ((acc.x ^ acc.y ^ acc.z ^ acc.w) == magic) *sink = acc;
}
}  // namespace ssd

extern "C" int ssd_read_probe(const void* buf, size_t bytes, int ctas_per_sm, void* sink, void* stream) {
  if (buf == nullptr || sink == nullptr || bytes < 16 || (bytes % 16) != 0) return SSD_ERR_INVALID;
  if (!ssd::aligned(buf, 16) || !ssd::aligned(sink, 16) || ctas_per_sm < 1 || ctas_per_sm > 8) return SSD_ERR_INVALID;
  const int dev = ssd::current_device();
  int sms = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return SSD_ERR_CUDA;
  ssd::k_read_probe<<<sms * ctas_per_sm, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(buf), bytes / 16, static_cast<uint4*>(sink), 0x9E3779B9u);
  ssd::count_launch();
  return ssd::check_launch();
}
