// C ABI of libcsa_gb300.so: argument validation, per-device facts, tensor-map
// encoding through the runtime's driver entry point, and the device status
// word that bounded waits report into. The compute lives in
// trimul_sm103a.cu and dense_sm103a.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "csa.h"
#include "csa_internal.h"

// Per device: [0] = first error code recorded by a kernel, [1] = wait site.
__device__ int g_csa_status[2];

namespace csa {
namespace {

thread_local std::string t_last_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int> g_inject{0};
std::atomic<int> g_dense_fetch{CSA_DENSE_FETCH_AUTO};
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

int set_error(int code, const std::string& msg) {
  t_last_error = msg;
  return code;
}

int cuda_error(const char* what, cudaError_t e) {
  return set_error(CSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace

int current_device(DeviceInfo& info, std::string& err) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return CSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    err = "device ordinal out of range";
    return CSA_ERR_CUDA;
  }
  // cudaGetDevice binds no context, and the tensor-map encoder is a driver
  // call that needs one: on a host thread that has made no runtime call that
  // touches the device yet, bind the device's primary context once.
  thread_local bool t_bound[kMaxDevices] = {};
  if (!t_bound[dev]) {
    if ((e = cudaSetDevice(dev)) != cudaSuccess) {
      err = std::string("cudaSetDevice: ") + cudaGetErrorString(e);
      return CSA_ERR_CUDA;
    }
    t_bound[dev] = true;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    d.device = dev;
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) ||
        (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev))) {
      err = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
      return CSA_ERR_CUDA;
    }
    d.cc = major * 10 + minor;
    if (d.cc != 103) {
      err = "this library is built for sm_103a (GB300); current device is sm_" +
            std::to_string(d.cc);
      return CSA_ERR_ARCH;
    }
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_csa_status)) != cudaSuccess) {
      err = std::string("cudaGetSymbolAddress(status): ") + cudaGetErrorString(e);
      return CSA_ERR_CUDA;
    }
    d.status_word = static_cast<int*>(p);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        err = "cuTensorMapEncodeTiled entry point unavailable";
        return CSA_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  info = g_dev[dev];
  return CSA_OK;
}

namespace {

// Per-stream SM limits (csa_set_stream_sm_limit): launches on a listed stream
// size their persistent grids and tilings for at most that many SMs.
struct SmLimit {
  cudaStream_t stream;
  int sms;
};
constexpr int kMaxSmLimits = 64;
std::mutex g_limit_mu;
SmLimit g_limits[kMaxSmLimits];
int g_limit_count = 0;
std::atomic<int> g_any_limit{0};

void apply_stream_sm_limit(DeviceInfo& info, cudaStream_t stream) {
  if (g_any_limit.load(std::memory_order_acquire) == 0) return;
  std::lock_guard<std::mutex> lock(g_limit_mu);
  for (int i = 0; i < g_limit_count; ++i)
    if (g_limits[i].stream == stream) {
      info.sm_count = std::max(1, std::min(info.sm_count, g_limits[i].sms));
      return;
    }
}

}  // namespace

namespace {

// Tensor maps are pure functions of their encoding parameters, so a map built
// once serves every later call with the same parameters (a buffer freed and
// reallocated at the same address with the same shape gets the same map).
// Direct-mapped cache of 256 entries, indexed by a hash of the parameters.
struct MapKey {
  uint64_t addr;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box[5];
  uint32_t dtype, rank, swizzle, pad;
};

struct MapEntry {
  bool valid = false;
  MapKey key{};
  CUtensorMap map{};
};

constexpr int kMapCacheSize = 256;
std::mutex g_map_mu;
MapEntry g_map_cache[kMapCacheSize];

uint64_t hash_key(const MapKey& k) {
  // FNV-1a over the key bytes.
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof k; ++i) h = (h ^ p[i]) * 1099511628211ull;
  return h;
}

std::mutex g_smem_mu;
struct SmemSetting {
  const void* fn;
  int device;
  int bytes;
};
SmemSetting g_smem_set[64];
int g_smem_count = 0;

}  // namespace

int set_max_dynamic_smem(const void* kernel, int bytes, int device, std::string& err) {
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (int i = 0; i < g_smem_count; ++i) {
    SmemSetting& e = g_smem_set[i];
    if (e.fn == kernel && e.device == device) {
      if (e.bytes >= bytes) return CSA_OK;
      cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (r != cudaSuccess) {
        err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(r);
        return CSA_ERR_LAUNCH;
      }
      e.bytes = bytes;
      return CSA_OK;
    }
  }
  cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(r);
    return CSA_ERR_LAUNCH;
  }
  if (g_smem_count < 64) g_smem_set[g_smem_count++] = SmemSetting{kernel, device, bytes};
  return CSA_OK;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* addr,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle, std::string& err) {
  MapKey key{};
  key.addr = reinterpret_cast<uint64_t>(addr);
  key.dtype = static_cast<uint32_t>(dtype);
  key.rank = rank;
  key.swizzle = static_cast<uint32_t>(swizzle);
  for (uint32_t i = 0; i < rank && i < 5; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  const int slot = static_cast<int>(hash_key(key) % kMapCacheSize);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    const MapEntry& e = g_map_cache[slot];
    if (e.valid && std::memcmp(&e.key, &key, sizeof key) == 0) {
      *map = e.map;
      return CSA_OK;
    }
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, rank, const_cast<void*>(addr), d, s, b, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    err = "cuTensorMapEncodeTiled failed (code " + std::to_string(static_cast<int>(r)) + ")";
    return CSA_ERR_ALIGN;
  }
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry& e = g_map_cache[slot];
    e.valid = true;
    e.key = key;
    e.map = *map;
  }
  return CSA_OK;
}

// The default bound: CSA_WAIT_LIMIT_NS from the environment when it holds a
// positive integer (read once), else 2 s.
uint64_t default_wait_limit_ns() {
  static const uint64_t v = [] {
    const char* e = std::getenv("CSA_WAIT_LIMIT_NS");
    if (e && *e) {
      char* end = nullptr;
      const unsigned long long x = std::strtoull(e, &end, 10);
      if (end && *end == '\0' && x > 0) return static_cast<uint64_t>(x);
    }
    return kDefaultWaitLimitNs;
  }();
  return v;
}

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load();
  return v ? v : default_wait_limit_ns();
}

namespace {

struct SlotFamily {
  bool ready = false;
  volatile unsigned long long* done_host = nullptr;  // page-locked, mapped: [kDirectSlots]
  unsigned long long* done_dev = nullptr;
  unsigned long long stream_id[kDirectSlots] = {};
  unsigned long long seq[kDirectSlots] = {};
  bool used[kDirectSlots] = {};
  int next_capture = 0;
  int cursor = 0;
  unsigned long long next_seq = 0;
};

std::mutex g_slot_mu;
SlotFamily g_slot_families[2][kMaxDevices];

}  // namespace

int acquire_counter_slot(int family, const DeviceInfo& dev, unsigned int* base, cudaStream_t stream,
                         CounterSlot& out, std::string& err) {
  if (family < 0 || family > 1 || dev.device < 0 || dev.device >= kMaxDevices || !base) {
    err = "counter slots: bad family or device";
    return CSA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_slot_mu);
  SlotFamily& f = g_slot_families[family][dev.device];
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) {
    err = std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e);
    return CSA_ERR_CUDA;
  }
  if (cs != cudaStreamCaptureStatusNone) {
    if (f.next_capture >= kCaptureSlots) {
      err = "more than " + std::to_string(kCaptureSlots) +
            " launches of this kernel captured into CUDA graphs in this process";
      return CSA_ERR_BUSY;
    }
    out.counters = base + kCounterWords * (kDirectSlots + f.next_capture++);
    out.done = nullptr;
    out.seq = 0;
    out.slot = -1;
    return CSA_OK;
  }
  // (made at the first launch outside capture: a captured launch needs none)
  if (!f.ready) {
    void* h = nullptr;
    e = cudaHostAlloc(&h, sizeof(unsigned long long) * kDirectSlots,
                      cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
      err = std::string("counter slots: page-locked completion words: ") + cudaGetErrorString(e);
      return CSA_ERR_CUDA;
    }
    std::memset(h, 0, sizeof(unsigned long long) * kDirectSlots);
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, h, 0);
    if (e != cudaSuccess) {
      cudaFreeHost(h);
      err = std::string("counter slots: cudaHostGetDevicePointer: ") + cudaGetErrorString(e);
      return CSA_ERR_CUDA;
    }
    f.done_host = static_cast<volatile unsigned long long*>(h);
    f.done_dev = static_cast<unsigned long long*>(d);
    f.ready = true;
  }
  unsigned long long sid = 0;
  e = cudaStreamGetId(stream, &sid);
  if (e != cudaSuccess) {
    err = std::string("cudaStreamGetId: ") + cudaGetErrorString(e);
    return CSA_ERR_CUDA;
  }
  int s = -1;
  for (int i = 0; i < kDirectSlots; ++i)
    if (f.used[i] && f.stream_id[i] == sid) {
      s = i;
      break;
    }
  if (s < 0) {
    for (int k = 0; k < kDirectSlots; ++k) {
      const int i = (f.cursor + k) % kDirectSlots;
      if (!f.used[i] || f.done_host[i] == f.seq[i]) {
        s = i;
        break;
      }
    }
    if (s < 0) {
      err = "launches on " + std::to_string(kDirectSlots) +
            " other streams are still in flight (work-list counter sets exhausted)";
      return CSA_ERR_BUSY;
    }
    f.cursor = (s + 1) % kDirectSlots;
    f.used[s] = true;
    f.stream_id[s] = sid;
  }
  f.seq[s] = ++f.next_seq;
  out.counters = base + kCounterWords * s;
  out.done = f.done_dev + s;
  out.seq = f.seq[s];
  out.slot = s;
  return CSA_OK;
}

void abandon_counter_slot(int family, const DeviceInfo& dev, const CounterSlot& slot) {
  if (slot.slot < 0 || family < 0 || family > 1 || dev.device < 0 || dev.device >= kMaxDevices)
    return;
  std::lock_guard<std::mutex> lock(g_slot_mu);
  SlotFamily& f = g_slot_families[family][dev.device];
  if (f.ready && f.seq[slot.slot] == slot.seq) f.done_host[slot.slot] = slot.seq;
}

bool take_inject() { return g_inject.exchange(0) != 0; }
int dense_fetch_mode() { return g_dense_fetch.load(); }

}  // namespace csa

using namespace csa;

// Checks shared by the dense entry points; CSA_OK or the status to return.
static int dense_args_ok(const char* who, const void* Y, const void* X, const void* W, int M,
                         int I, int H) {
  if (!Y || !X || !W) return set_error(CSA_ERR_NULL, std::string(who) + ": null pointer");
  if (M <= 0 || I <= 0 || H <= 0)
    return set_error(CSA_ERR_SHAPE, std::string(who) + ": M, I, H must be >= 1");
  if (reinterpret_cast<uintptr_t>(X) % 2 || reinterpret_cast<uintptr_t>(W) % 2 ||
      reinterpret_cast<uintptr_t>(Y) % 4)
    return set_error(CSA_ERR_ALIGN, std::string(who) + ": X, W need 2-byte and Y 4-byte alignment");
  return CSA_OK;
}

extern "C" {

csa_status trimul_forward_ex(float* out, const void* qkv, int B, int T, int C, int NH,
                             uint32_t mask_bits, uint32_t flags, void* stream) {
  t_last_error.clear();
  if (!out || !qkv) return set_error(CSA_ERR_NULL, "trimul_forward: null pointer");
  if (B <= 0 || T <= 0 || C <= 0 || NH <= 0)
    return set_error(CSA_ERR_SHAPE, "trimul_forward: B, T, C, NH must be >= 1");
  if (C % NH != 0) return set_error(CSA_ERR_SHAPE, "trimul_forward: C % NH != 0");
  if (flags & ~CSA_TRIMUL_LOWER_ONLY)
    return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward: unknown flags");
  const int HS = C / NH;
  if (HS % 8 != 0)
    return set_error(CSA_ERR_ALIGN, "trimul_forward: HS = C/NH must be a multiple of 8");
  if (HS > 256) return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward: HS > 256");
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return set_error(CSA_ERR_ALIGN, "trimul_forward: qkv must be 16-byte aligned, out 4-byte");
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = trimul_launch(out, qkv, B, T, C, NH, mask_bits, flags, static_cast<cudaStream_t>(stream),
                     dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status trimul_forward_f32(float* out, const float* qkv, int B, int T, int C, int NH,
                              uint32_t mask_bits, uint32_t flags, void* stream) {
  t_last_error.clear();
  if (!out || !qkv) return set_error(CSA_ERR_NULL, "trimul_forward_f32: null pointer");
  if (B <= 0 || T <= 0 || C <= 0 || NH <= 0)
    return set_error(CSA_ERR_SHAPE, "trimul_forward_f32: B, T, C, NH must be >= 1");
  if (C % NH != 0) return set_error(CSA_ERR_SHAPE, "trimul_forward_f32: C % NH != 0");
  if (flags & ~CSA_TRIMUL_LOWER_ONLY)
    return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward_f32: unknown flags");
  const int HS = C / NH;
  if (HS % 4 != 0)
    return set_error(CSA_ERR_ALIGN, "trimul_forward_f32: HS = C/NH must be a multiple of 4");
  if (HS > 256) return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward_f32: HS > 256");
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return set_error(CSA_ERR_ALIGN, "trimul_forward_f32: qkv must be 16-byte aligned, out 4-byte");
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = trimul_f32_launch(out, qkv, B, T, C, NH, mask_bits, flags,
                         static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status trimul_forward_noalloc(float* out, const void* qkv, int B, int T, int C, int NH,
                                  uint32_t mask_bits, uint32_t flags, void* stream) {
  t_last_error.clear();
  if (!out || !qkv) return set_error(CSA_ERR_NULL, "trimul_forward_noalloc: null pointer");
  if (B <= 0 || T <= 0 || C <= 0 || NH <= 0)
    return set_error(CSA_ERR_SHAPE, "trimul_forward_noalloc: B, T, C, NH must be >= 1");
  if (C % NH != 0) return set_error(CSA_ERR_SHAPE, "trimul_forward_noalloc: C % NH != 0");
  if (flags & ~CSA_TRIMUL_LOWER_ONLY)
    return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward_noalloc: unknown flags");
  const int HS = C / NH;
  if (HS % 8 != 0)
    return set_error(CSA_ERR_ALIGN, "trimul_forward_noalloc: HS = C/NH must be a multiple of 8");
  if (HS > 256) return set_error(CSA_ERR_UNSUPPORTED, "trimul_forward_noalloc: HS > 256");
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return set_error(CSA_ERR_ALIGN,
                     "trimul_forward_noalloc: qkv must be 16-byte aligned, out 4-byte");
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = trimul_launch_noalloc(out, qkv, B, T, C, NH, mask_bits, flags,
                             static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status trimul_forward(float* out, const void* qkv, int B, int T, int C, int NH) {
  return trimul_forward_ex(out, qkv, B, T, C, NH, CSA_MASK_NAN, CSA_TRIMUL_FULL, nullptr);
}

csa_status causal_softmax_forward(float* att, const void* qkv, int B, int T, int C, int NH,
                                  void* stream) {
  t_last_error.clear();
  if (!att || !qkv) return set_error(CSA_ERR_NULL, "causal_softmax_forward: null pointer");
  if (B <= 0 || T <= 0 || C <= 0 || NH <= 0)
    return set_error(CSA_ERR_SHAPE, "causal_softmax_forward: B, T, C, NH must be >= 1");
  if (C % NH != 0) return set_error(CSA_ERR_SHAPE, "causal_softmax_forward: C % NH != 0");
  const int HS = C / NH;
  if (HS % 8 != 0)
    return set_error(CSA_ERR_ALIGN, "causal_softmax_forward: HS = C/NH must be a multiple of 8");
  if (HS > 128) return set_error(CSA_ERR_UNSUPPORTED, "causal_softmax_forward: HS > 128");
  if (reinterpret_cast<uintptr_t>(qkv) % 16 != 0 || reinterpret_cast<uintptr_t>(att) % 4 != 0)
    return set_error(CSA_ERR_ALIGN,
                     "causal_softmax_forward: qkv must be 16-byte aligned, att 4-byte");
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = softmax_launch(att, qkv, B, T, C, NH, static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status batch_matmul_nt(float* Y, const void* X, const void* W, int batch, int T1, int T2,
                           int D, void* stream) {
  t_last_error.clear();
  if (!Y || !X || !W) return set_error(CSA_ERR_NULL, "batch_matmul_nt: null pointer");
  if (batch <= 0 || T1 <= 0 || T2 <= 0 || D <= 0)
    return set_error(CSA_ERR_SHAPE, "batch_matmul_nt: batch, T1, T2, D must be >= 1");
  if (D % 8 != 0)
    return set_error(CSA_ERR_ALIGN, "batch_matmul_nt: D must be a multiple of 8");
  if (D > 256) return set_error(CSA_ERR_UNSUPPORTED, "batch_matmul_nt: D > 256");
  if (reinterpret_cast<uintptr_t>(X) % 16 || reinterpret_cast<uintptr_t>(W) % 16 ||
      reinterpret_cast<uintptr_t>(Y) % 4)
    return set_error(CSA_ERR_ALIGN, "batch_matmul_nt: X, W need 16-byte and Y 4-byte alignment");
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = bmm_nt_launch(Y, X, W, batch, T1, T2, D, static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status dense_xwt_ex(float* Y, const void* X, const void* W, int M, int I, int H,
                        void* stream) {
  t_last_error.clear();
  int rc = dense_args_ok("dense_xwt", Y, X, W, M, I, H);
  if (rc != CSA_OK) return rc;
  DeviceInfo dev;
  std::string err;
  rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = dense_launch(Y, X, W, M, I, H, nullptr, 0, static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status dense_xwt_workspace_size(const void* X, const void* W, int M, int I, int H,
                                    size_t* bytes) {
  t_last_error.clear();
  if (!bytes) return set_error(CSA_ERR_NULL, "dense_xwt_workspace_size: null pointer");
  *bytes = 0;
  if (!X || !W) return set_error(CSA_ERR_NULL, "dense_xwt_workspace_size: null pointer");
  if (M <= 0 || I <= 0 || H <= 0)
    return set_error(CSA_ERR_SHAPE, "dense_xwt_workspace_size: M, I, H must be >= 1");
  *bytes = dense_workspace_bytes(X, W, M, I, H);
  return CSA_OK;
}

csa_status dense_xwt_ws(float* Y, const void* X, const void* W, int M, int I, int H,
                        void* workspace, size_t workspace_bytes, void* stream) {
  t_last_error.clear();
  int rc = dense_args_ok("dense_xwt_ws", Y, X, W, M, I, H);
  if (rc != CSA_OK) return rc;
  const size_t need = dense_workspace_bytes(X, W, M, I, H);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return set_error(CSA_ERR_WORKSPACE, "dense_xwt_ws: " + std::to_string(need) +
                                            " bytes of workspace needed, " +
                                            std::to_string(workspace ? workspace_bytes : 0) +
                                            " given");
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return set_error(CSA_ERR_ALIGN, "dense_xwt_ws: workspace must be 16-byte aligned");
  DeviceInfo dev;
  std::string err;
  rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = dense_launch(Y, X, W, M, I, H, need > 0 ? workspace : nullptr, workspace_bytes,
                    static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status dense_xwt(float* Y, const void* X, const void* W, int M, int I, int H) {
  return dense_xwt_ex(Y, X, W, M, I, H, nullptr);
}

// Checks shared by the grouped dense entry points; CSA_OK or the status to return.
static int grouped_args_ok(const char* who, float* const* Y, const void* const* X, const void* W,
                           const int* M, int n, int I, int H) {
  if (!Y || !X || !W || !M) return set_error(CSA_ERR_NULL, std::string(who) + ": null pointer");
  if (n <= 0 || I <= 0 || H <= 0)
    return set_error(CSA_ERR_SHAPE, std::string(who) + ": n, I, H must be >= 1");
  if (reinterpret_cast<uintptr_t>(W) % 2)
    return set_error(CSA_ERR_ALIGN, std::string(who) + ": W needs 2-byte alignment");
  for (int g = 0; g < n; ++g) {
    if (!Y[g] || !X[g])
      return set_error(CSA_ERR_NULL, std::string(who) + ": null pointer in problem " +
                                         std::to_string(g));
    if (M[g] <= 0)
      return set_error(CSA_ERR_SHAPE, std::string(who) + ": M[" + std::to_string(g) +
                                          "] must be >= 1");
    if (reinterpret_cast<uintptr_t>(X[g]) % 2 || reinterpret_cast<uintptr_t>(Y[g]) % 4)
      return set_error(CSA_ERR_ALIGN, std::string(who) + ": X[" + std::to_string(g) +
                                          "] needs 2-byte and Y 4-byte alignment");
  }
  return CSA_OK;
}

csa_status dense_xwt_grouped_ws(float* const* Y, const void* const* X, const void* W,
                                const int* M, int n, int I, int H, void* workspace,
                                size_t workspace_bytes, void* stream) {
  t_last_error.clear();
  int rc = grouped_args_ok("dense_xwt_grouped", Y, X, W, M, n, I, H);
  if (rc != CSA_OK) return rc;
  if (workspace) {
    const size_t need = dense_grouped_workspace_bytes(X, W, M, n, I, H);
    if (workspace_bytes < need)
      return set_error(CSA_ERR_WORKSPACE, "dense_xwt_grouped_ws: " + std::to_string(need) +
                                              " bytes of workspace needed, " +
                                              std::to_string(workspace_bytes) + " given");
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
      return set_error(CSA_ERR_ALIGN, "dense_xwt_grouped_ws: workspace must be 16-byte aligned");
  }
  DeviceInfo dev;
  std::string err;
  rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  apply_stream_sm_limit(dev, static_cast<cudaStream_t>(stream));
  rc = dense_grouped_launch(Y, X, W, M, n, I, H, workspace, workspace_bytes,
                            static_cast<cudaStream_t>(stream), dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  return CSA_OK;
}

csa_status dense_xwt_grouped(float* const* Y, const void* const* X, const void* W, const int* M,
                             int n, int I, int H, void* stream) {
  return dense_xwt_grouped_ws(Y, X, W, M, n, I, H, nullptr, 0, stream);
}

csa_status dense_xwt_grouped_workspace_size(const void* const* X, const void* W, const int* M,
                                            int n, int I, int H, size_t* bytes) {
  t_last_error.clear();
  if (!bytes) return set_error(CSA_ERR_NULL, "dense_xwt_grouped_workspace_size: null pointer");
  *bytes = 0;
  if (!X || !W || !M) return set_error(CSA_ERR_NULL, "dense_xwt_grouped_workspace_size: null pointer");
  if (n <= 0 || I <= 0 || H <= 0)
    return set_error(CSA_ERR_SHAPE, "dense_xwt_grouped_workspace_size: n, I, H must be >= 1");
  for (int g = 0; g < n; ++g) {
    if (!X[g]) return set_error(CSA_ERR_NULL, "dense_xwt_grouped_workspace_size: null pointer");
    if (M[g] <= 0)
      return set_error(CSA_ERR_SHAPE, "dense_xwt_grouped_workspace_size: M[g] must be >= 1");
  }
  *bytes = dense_grouped_workspace_bytes(X, W, M, n, I, H);
  return CSA_OK;
}

csa_status csa_get_status(void* stream) {
  t_last_error.clear();
  DeviceInfo dev;
  std::string err;
  int rc = current_device(dev, err);
  if (rc != CSA_OK) return set_error(rc, err);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error("csa_get_status: cudaStreamSynchronize", e);
  int host[2] = {0, 0};
  e = cudaMemcpy(host, dev.status_word, sizeof host, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error("csa_get_status: read status", e);
  if (host[0] != 0) {
    const int zero[2] = {0, 0};
    e = cudaMemcpy(dev.status_word, zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_error("csa_get_status: clear status", e);
    t_last_error = "device wait ran out at site " + std::to_string(host[1]);
    return host[0];
  }
  return CSA_OK;
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_NULL: return "null pointer";
    case CSA_ERR_SHAPE: return "invalid shape";
    case CSA_ERR_ALIGN: return "alignment or stride requirement not met";
    case CSA_ERR_UNSUPPORTED: return "unsupported size or flag";
    case CSA_ERR_ARCH: return "device is not sm_103";
    case CSA_ERR_LAUNCH: return "kernel launch failed";
    case CSA_ERR_TIMEOUT: return "device-side wait ran out";
    case CSA_ERR_CUDA: return "CUDA call failed";
    case CSA_ERR_CHECK: return "device-side index check failed (debug build)";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_BUSY: return "work-list counter sets exhausted";
    default: return "unknown status";
  }
}

const char* csa_last_error(void) { return t_last_error.c_str(); }

const char* csa_version(void) { return "0.1.0 sm_103a"; }

void csa_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }

uint64_t csa_get_wait_limit_ns(void) { return csa::wait_limit_ns(); }

void csa_debug_inject(int enable) { g_inject.store(enable ? 1 : 0); }

}  // extern "C"

namespace {

// Streams held by csa_debug_hold_stream: each hold is a host function that
// waits for its release (or 10 s) on the CUDA runtime's callback thread.
std::mutex g_hold_mu;
std::condition_variable g_hold_cv;
unsigned long long g_hold_issued = 0, g_hold_released = 0;

void CUDART_CB hold_stream_fn(void* arg) {
  const unsigned long long gen = static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(arg));
  std::unique_lock<std::mutex> lock(g_hold_mu);
  g_hold_cv.wait_for(lock, std::chrono::seconds(10), [&] { return g_hold_released >= gen; });
}

}  // namespace

extern "C" {

csa_status csa_debug_hold_stream(void* stream) {
  t_last_error.clear();
  unsigned long long gen;
  {
    std::lock_guard<std::mutex> lock(g_hold_mu);
    gen = ++g_hold_issued;
  }
  cudaError_t e = cudaLaunchHostFunc(static_cast<cudaStream_t>(stream), hold_stream_fn,
                                     reinterpret_cast<void*>(static_cast<uintptr_t>(gen)));
  if (e != cudaSuccess) return cuda_error("csa_debug_hold_stream", e);
  return CSA_OK;
}

void csa_debug_release_streams(void) {
  {
    std::lock_guard<std::mutex> lock(g_hold_mu);
    g_hold_released = g_hold_issued;
  }
  g_hold_cv.notify_all();
}

csa_status csa_dense_tiling(int M, int H, int sms, int* bn, int* pairs) {
  t_last_error.clear();
  if (!bn || !pairs) return set_error(CSA_ERR_NULL, "csa_dense_tiling: null pointer");
  if (M <= 0 || H <= 0 || sms <= 0)
    return set_error(CSA_ERR_SHAPE, "csa_dense_tiling: M, H, sms must be >= 1");
  int b = 0;
  bool p = false;
  dense_tiling(M, H, sms, true, b, p);
  *bn = b;
  *pairs = p ? 1 : 0;
  return CSA_OK;
}

csa_status csa_set_stream_sm_limit(void* stream, int max_sms) {
  t_last_error.clear();
  if (max_sms < 0)
    return set_error(CSA_ERR_SHAPE, "csa_set_stream_sm_limit: max_sms must be >= 0");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_limit_mu);
  for (int i = 0; i < g_limit_count; ++i) {
    if (g_limits[i].stream != s) continue;
    if (max_sms == 0) {
      g_limits[i] = g_limits[--g_limit_count];
    } else {
      g_limits[i].sms = max_sms;
    }
    g_any_limit.store(g_limit_count, std::memory_order_release);
    return CSA_OK;
  }
  if (max_sms == 0) return CSA_OK;
  if (g_limit_count == kMaxSmLimits)
    return set_error(CSA_ERR_BUSY, "csa_set_stream_sm_limit: 64 streams already carry a limit");
  g_limits[g_limit_count++] = SmLimit{s, max_sms};
  g_any_limit.store(g_limit_count, std::memory_order_release);
  return CSA_OK;
}

csa_status csa_get_stream_sm_limit(void* stream, int* max_sms) {
  t_last_error.clear();
  if (!max_sms) return set_error(CSA_ERR_NULL, "csa_get_stream_sm_limit: null pointer");
  *max_sms = 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_limit_mu);
  for (int i = 0; i < g_limit_count; ++i)
    if (g_limits[i].stream == s) *max_sms = g_limits[i].sms;
  return CSA_OK;
}

csa_status csa_set_dense_fetch(int mode) {
  if (mode != CSA_DENSE_FETCH_AUTO && mode != CSA_DENSE_FETCH_LOADERS)
    return set_error(CSA_ERR_SHAPE, "csa_set_dense_fetch: unknown mode " + std::to_string(mode));
  g_dense_fetch.store(mode);
  return CSA_OK;
}

}  // extern "C"
