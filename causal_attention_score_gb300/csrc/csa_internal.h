// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "csa.h"

namespace csa {

// Per-device facts, queried once per device and cached.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc = 0;              // major * 10 + minor
  int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
  int* status_word = nullptr;  // device address of the [code, site] status pair
};

// Fills `info` for the current device. Returns CSA_OK, CSA_ERR_CUDA or CSA_ERR_ARCH.
int current_device(DeviceInfo& info, std::string& err);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link),
// with a cache of maps keyed by every encoding parameter.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* addr,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle, std::string& err);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel, device and
// larger size; later calls needing no more are free.
int set_max_dynamic_smem(const void* kernel, int bytes, int device, std::string& err);

// Launches `kernel` with programmatic stream serialization: it may start while
// the previous kernel in the stream finishes, and waits for it (griddepcontrol)
// before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// launch_programmatic with clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                        size_t smem, cudaStream_t stream, unsigned cluster_x,
                                        Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------- work-list counter slots --
//
// The score and softmax kernels take work-list positions from a set of global
// counters that the last CTA of each launch resets to zero. Two launches may
// share a set only if they never run at the same time. Each kernel family keeps
// kDirectSlots + kCaptureSlots sets per device (a fixed device array) and hands
// them out as follows:
//  - a launch outside stream capture uses its stream's set: launches on one
//    stream run in order. A stream's set is taken from a set whose last launch
//    has signalled completion (the kernel's last CTA writes the launch's number
//    into page-locked host memory) or that was never used; when all direct sets
//    belong to streams with launches in flight, the call fails with CSA_ERR_BUSY;
//  - a launch captured into a CUDA graph gets a set of its own for good (the
//    graph may be replayed at any time, next to anything else): at most
//    kCaptureSlots captured launches per kernel family and process.
constexpr int kCounterWords = 4;
constexpr int kDirectSlots = 256;
constexpr int kCaptureSlots = 1024;
enum CounterFamily : int { kFamilyScores = 0, kFamilySoftmax = 1 };

struct CounterSlot {
  unsigned int* counters = nullptr;  // the set (kCounterWords words), zero at launch
  unsigned long long* done = nullptr;  // device address of its completion word (nullptr: none)
  unsigned long long seq = 0;          // number the launch writes there when it completes
  int slot = -1;                       // direct slot index, -1 for a captured set
};

// The set for a launch on `stream`; `base` is the family's device array of
// (kDirectSlots + kCaptureSlots) * kCounterWords words.
int acquire_counter_slot(int family, const DeviceInfo& dev, unsigned int* base, cudaStream_t stream,
                         CounterSlot& out, std::string& err);
// A launch given `slot` failed: its set is free again.
void abandon_counter_slot(int family, const DeviceInfo& dev, const CounterSlot& slot);

// Bound (ns of %globaltimer) on every mbarrier/flag wait in the kernels.
uint64_t wait_limit_ns();
// True once after csa_debug_inject armed it: the next launch withholds one arrival.
bool take_inject();
// The dense layer's fetch mode set by csa_set_dense_fetch (CSA_DENSE_FETCH_*).
int dense_fetch_mode();

// Kernel launchers; each validates what is specific to its kernel.
// `counters`: work-list counter pair to use instead of the library's per-launch
// slot ring (nullptr = slot ring); it must be zero when the kernel starts.
int trimul_launch(float* out, const void* qkv, int B, int T, int C, int NH, uint32_t mask_bits,
                  uint32_t flags, cudaStream_t stream, const DeviceInfo& dev, std::string& err,
                  unsigned int* counters = nullptr);

// trimul_launch with its scratch in a fixed device array (no allocation).
int trimul_launch_noalloc(float* out, const void* qkv, int B, int T, int C, int NH,
                          uint32_t mask_bits, uint32_t flags, cudaStream_t stream,
                          const DeviceInfo& dev, std::string& err);

int trimul_f32_launch(float* out, const float* qkv, int B, int T, int C, int NH,
                      uint32_t mask_bits, uint32_t flags, cudaStream_t stream, const DeviceInfo& dev,
                      std::string& err);
int bmm_nt_launch(float* Y, const void* X, const void* W, int batch, int T1, int T2, int D,
                  cudaStream_t stream, const DeviceInfo& dev, std::string& err);

int softmax_launch(float* out, const void* qkv, int B, int T, int C, int NH, cudaStream_t stream,
                   const DeviceInfo& dev, std::string& err);

// One dense layer. Rows no tensor map can describe are first copied into
// `workspace` (ws_bytes long, at least dense_workspace_bytes) as 16-byte-aligned
// rows, or fetched by loader warps when workspace is nullptr.
int dense_launch(float* Y, const void* X, const void* W, int M, int I, int H, void* workspace,
                 size_t ws_bytes, cudaStream_t stream, const DeviceInfo& dev, std::string& err);

// Workspace bytes dense_launch needs to realign X and W (0 when their rows need none).
// The tile width (64..256) and form (CTA pairs or single CTAs) that one problem of
// M rows and H columns takes on `sms` SMs when clusters of two fit; pairs need rows
// fetched by TMA (tma_rows).
void dense_tiling(int M, int H, int sms, bool tma_rows, int& bn, bool& pair);

size_t dense_workspace_bytes(const void* X, const void* W, int M, int I, int H);

// Dense layers sharing W. Rows no tensor map can describe are first copied into
// `workspace` (at least dense_grouped_workspace_bytes), or each problem runs as its
// own loader-warp dense_launch when workspace is nullptr.
int dense_grouped_launch(float* const* Y, const void* const* X, const void* W, const int* M, int n,
                         int I, int H, void* workspace, size_t ws_bytes, cudaStream_t stream,
                         const DeviceInfo& dev, std::string& err);
size_t dense_grouped_workspace_bytes(const void* const* X, const void* W, const int* M, int n,
                                     int I, int H);

}  // namespace csa
