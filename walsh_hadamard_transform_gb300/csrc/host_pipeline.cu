// Host-buffer entry points: copy in, transform, copy out, as a three-stage
// pipeline over chunks of whole vectors.
//
// The batch is cut into chunks of c vectors.  A caller-provided device workspace
// holds up to three chunks (slots).  Chunk k is copied host -> device on the
// library's copy-in stream, transformed in place on the caller's stream, and
// copied device -> host on the copy-out stream; events order the three stages of
// one chunk and keep a slot from being refilled before its previous chunk has
// left.  So the host -> device copy of chunk k+1, the transform of chunk k and the
// device -> host copy of chunk k-1 run at the same time, and both directions of
// the host link are busy at once.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fwt.h"
#include "registry.cuh"

namespace fwt {
namespace {

constexpr int kSlots = 3;
constexpr size_t kSlotAlign = 256;          // slot parts start on 256-byte boundaries
constexpr size_t kTargetChunkBytes = 32ull << 20;  // smallest chunk worth a pipeline stage
constexpr int64_t kTargetChunks = 16;

struct DeviceStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t joined_in = nullptr, joined_out = nullptr;  // error path: copy streams -> caller
  cudaEvent_t loaded[kSlots] = {}, done[kSlots] = {}, drained[kSlots] = {};
};

std::mutex g_mu;
std::vector<DeviceStreams> g_dev;

cudaError_t streams_for_current_device(DeviceStreams*& ds) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
  ds = &g_dev[dev];
  if (ds->ready) return cudaSuccess;
  err = cudaStreamCreateWithFlags(&ds->in, cudaStreamNonBlocking);
  if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&ds->out, cudaStreamNonBlocking);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ds->start, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ds->joined_in, cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ds->joined_out, cudaEventDisableTiming);
  for (int s = 0; s < kSlots && err == cudaSuccess; ++s) {
    err = cudaEventCreateWithFlags(&ds->loaded[s], cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ds->done[s], cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&ds->drained[s], cudaEventDisableTiming);
  }
  if (err == cudaSuccess) ds->ready = true;
  return err;
}

size_t align_up(size_t v) { return (v + kSlotAlign - 1) / kSlotAlign * kSlotAlign; }

// Bytes of one slot holding c vectors of `parts` arrays.
size_t slot_bytes(int esz, int n, int64_t c, int parts) {
  return (size_t)parts * align_up((size_t)(c << n) * (size_t)esz);
}

// Vectors a chunk should hold: about batch / 16, at least 32 MiB, at most the batch.
int64_t target_chunk(int esz, int n, int64_t batch, int parts) {
  const size_t vec = (size_t)parts * ((size_t)1 << n) * (size_t)esz;
  int64_t c = (batch + kTargetChunks - 1) / kTargetChunks;
  c = std::max<int64_t>(c, (int64_t)((kTargetChunkBytes + vec - 1) / vec));
  return std::max<int64_t>(1, std::min(c, batch));
}

// How a call's batch is cut into chunks and slots, from its arguments alone.
struct HostPlan {
  int esz = 4;
  bool has_im = false;
  int64_t c = 0;        // vectors per chunk
  size_t sb = 0;        // bytes of one slot (both parts)
  size_t part_off = 0;  // offset of the imaginary part within a slot
  int slots = 0;
};

// Every argument check of a host-buffer call, before any CUDA call: sizes, the
// pointers (the workspace pointer itself is checked by the caller), overlapping
// host arrays, and whether one vector fits `workspace_bytes`.  FWT_OK with
// batch == 0 means there is nothing to do.
int validate_host(int dtype, const void* re_in, const void* im_in, const void* re_out,
                  const void* im_out, int n, int64_t batch, int normalize,
                  size_t workspace_bytes, HostPlan& hp) {
  if (n < 0 || n > 30 || batch < 0) return FWT_ERR_INVALID_ARG;
  if (batch == 0) return FWT_OK;
  const int esz = dtype == FWT_C64 ? 8 : 4;
  if (batch > (INT64_MAX >> n) / esz) return FWT_ERR_INVALID_ARG;
  if (!re_in || !re_out) return FWT_ERR_INVALID_ARG;
  const bool has_im = im_in || im_out;
  if (has_im && (!im_in || !im_out)) return FWT_ERR_INVALID_ARG;
  if (!has_im && dtype != FWT_I32) return FWT_ERR_INVALID_ARG;
  if (dtype == FWT_I32 && normalize) return FWT_ERR_UNSUPPORTED;
  const size_t bytes = (size_t)(batch << n) * (size_t)esz;
  // host outputs may coincide exactly with their own input, and with nothing else
  auto disjoint = [bytes](const void* a, const void* b) {
    return (uintptr_t)a + bytes <= (uintptr_t)b || (uintptr_t)b + bytes <= (uintptr_t)a;
  };
  if (re_out != re_in && !disjoint(re_out, re_in)) return FWT_ERR_INVALID_ARG;
  if (has_im) {
    if (im_out != im_in && !disjoint(im_out, im_in)) return FWT_ERR_INVALID_ARG;
    if (!disjoint(re_out, im_out) || !disjoint(re_out, im_in) || !disjoint(im_out, re_in))
      return FWT_ERR_INVALID_ARG;
  }
  const int parts = has_im ? 2 : 1;
  // chunk size and slot count from the workspace
  int64_t c = target_chunk(esz, n, batch, parts);
  while (c > 1 && slot_bytes(esz, n, c, parts) * kSlots > workspace_bytes) c = (c + 1) / 2;
  const size_t sb = slot_bytes(esz, n, c, parts);
  const int slots = (int)std::min<size_t>(kSlots, workspace_bytes / sb);
  if (slots < 1) return FWT_ERR_INVALID_ARG;  // not even one vector fits
  hp.esz = esz;
  hp.has_im = has_im;
  hp.c = c;
  hp.sb = sb;
  hp.part_off = align_up((size_t)(c << n) * (size_t)esz);
  hp.slots = slots;
  return FWT_OK;
}

// Enqueues the pipeline of a validated call (batch > 0).  `started` becomes true
// once anything has been enqueued.  On a failure after that, the two copy streams
// are joined back into `stream` (best effort), so that work the caller enqueues on
// `stream` afterwards still comes after every copy this call enqueued.
int enqueue_host(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out,
                 int n, int64_t batch, int normalize, void* workspace, const HostPlan& hp,
                 cudaStream_t stream, bool& started) {
  started = false;
  const int esz = hp.esz;
  const bool has_im = hp.has_im;
  const int64_t c = hp.c;
  const int slots = hp.slots;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceStreams* ds = nullptr;
  cudaError_t err = streams_for_current_device(ds);
  if (err != cudaSuccess) {
    set_last_cuda_error((int)err);
    return FWT_ERR_CUDA;
  }
  auto fail = [&](int status, cudaError_t e) {
    if (status == FWT_ERR_CUDA) set_last_cuda_error((int)e);
    if (started) {
      if (cudaEventRecord(ds->joined_in, ds->in) == cudaSuccess)
        cudaStreamWaitEvent(stream, ds->joined_in, 0);
      if (cudaEventRecord(ds->joined_out, ds->out) == cudaSuccess)
        cudaStreamWaitEvent(stream, ds->joined_out, 0);
    }
    return status;
  };
  // nothing starts before the work the caller enqueued on `stream` so far
  err = cudaEventRecord(ds->start, stream);
  if (err != cudaSuccess) return fail(FWT_ERR_CUDA, err);
  started = true;
  err = cudaStreamWaitEvent(ds->in, ds->start, 0);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(ds->out, ds->start, 0);
  if (err != cudaSuccess) return fail(FWT_ERR_CUDA, err);

  const int64_t chunks = (batch + c - 1) / c;
  for (int64_t k = 0; k < chunks; ++k) {
    const int s = (int)(k % slots);
    const int64_t v0 = k * c, nv = std::min(c, batch - v0);
    const size_t off = (size_t)(v0 << n) * (size_t)esz, len = (size_t)(nv << n) * (size_t)esz;
    char* d_re = (char*)workspace + (size_t)s * hp.sb;
    char* d_im = has_im ? d_re + hp.part_off : nullptr;
    // copy in, once the slot's previous chunk has been copied out
    if (k >= slots) err = cudaStreamWaitEvent(ds->in, ds->drained[s], 0);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(d_re, (const char*)re_in + off, len, cudaMemcpyHostToDevice, ds->in);
    if (err == cudaSuccess && has_im)
      err = cudaMemcpyAsync(d_im, (const char*)im_in + off, len, cudaMemcpyHostToDevice, ds->in);
    if (err == cudaSuccess) err = cudaEventRecord(ds->loaded[s], ds->in);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(stream, ds->loaded[s], 0);
    if (err != cudaSuccess) return fail(FWT_ERR_CUDA, err);
    // transform in place on the caller's stream
    int st;
    if (dtype == FWT_C32)
      st = fwt_batched_c32((const float*)d_re, (const float*)d_im, (float*)d_re, (float*)d_im, n,
                           nv, normalize, stream);
    else if (dtype == FWT_C64)
      st = fwt_batched_c64((const double*)d_re, (const double*)d_im, (double*)d_re,
                           (double*)d_im, n, nv, normalize, stream);
    else
      st = fwt_batched_i32((const int32_t*)d_re, (const int32_t*)d_im, (int32_t*)d_re,
                           (int32_t*)d_im, n, nv, 0, stream);
    if (st != FWT_OK) return fail(st, cudaSuccess);  // the transform recorded its own error
    err = cudaEventRecord(ds->done[s], stream);
    // copy out
    if (err == cudaSuccess) err = cudaStreamWaitEvent(ds->out, ds->done[s], 0);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync((char*)re_out + off, d_re, len, cudaMemcpyDeviceToHost, ds->out);
    if (err == cudaSuccess && has_im)
      err = cudaMemcpyAsync((char*)im_out + off, d_im, len, cudaMemcpyDeviceToHost, ds->out);
    if (err == cudaSuccess) err = cudaEventRecord(ds->drained[s], ds->out);
    if (err != cudaSuccess) return fail(FWT_ERR_CUDA, err);
  }
  // the caller's stream reaches this point only after the last copy out
  err = cudaStreamWaitEvent(stream, ds->drained[(chunks - 1) % slots], 0);
  return err == cudaSuccess ? FWT_OK : fail(FWT_ERR_CUDA, err);
}

int run_host(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out, int n,
             int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
             cudaStream_t stream) {
  HostPlan hp;
  int st = validate_host(dtype, re_in, im_in, re_out, im_out, n, batch, normalize,
                         workspace_bytes, hp);
  if (st != FWT_OK || batch == 0) return st;
  if (!workspace) return FWT_ERR_INVALID_ARG;
  if ((uintptr_t)workspace & 15u) return FWT_ERR_MISALIGNED;
  bool started = false;
  return enqueue_host(dtype, re_in, im_in, re_out, im_out, n, batch, normalize, workspace, hp,
                      stream, started);
}

}  // namespace
}  // namespace fwt

extern "C" {

size_t fwt_host_workspace_bytes(int dtype, int n, int64_t batch, int with_im) {
  if (dtype < 0 || dtype > 2 || n < 0 || n > 30 || batch <= 0) return 0;
  const int esz = dtype == FWT_C64 ? 8 : 4;
  const int parts = (with_im || dtype != FWT_I32) ? 2 : 1;
  const int64_t c = fwt::target_chunk(esz, n, batch, parts);
  const int64_t chunks = (batch + c - 1) / c;
  return fwt::slot_bytes(esz, n, c, parts) * (size_t)std::min<int64_t>(fwt::kSlots, chunks);
}

int fwt_host_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream) {
  return fwt::run_host(FWT_C32, re_in, im_in, re_out, im_out, n, batch, normalize, workspace,
                       workspace_bytes, (cudaStream_t)stream);
}

int fwt_host_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream) {
  return fwt::run_host(FWT_C64, re_in, im_in, re_out, im_out, n, batch, normalize, workspace,
                       workspace_bytes, (cudaStream_t)stream);
}

int fwt_host_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream) {
  return fwt::run_host(FWT_I32, re_in, im_in, re_out, im_out, n, batch, normalize, workspace,
                       workspace_bytes, (cudaStream_t)stream);
}

}  // extern "C"

// ---- host-buffer entry points with a static device workspace -------------------------
// The same pipeline over a workspace that is part of the module image: a file-scope
// device array (allocated with the module when it loads, one per device), found with
// cudaGetSymbolAddress.  The library allocates nothing at run time.  Calls share the
// buffer, so each one first waits (on the caller's stream) for the previous one to
// have copied its last chunk out.  The buffer's address and that event are looked up
// once per device and kept: they do not survive cudaDeviceReset or the destruction
// of the device's primary context (nor do the copy streams above).
namespace fwt {
namespace {

constexpr size_t kStaticWorkspaceBytes = 512ull << 20;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

struct StaticWorkspace {
  void* ptr = nullptr;
  cudaEvent_t done = nullptr;  // recorded on the caller's stream after each call
  bool used = false;
};
std::mutex g_static_mu;  // taken before g_mu, never after it
std::vector<StaticWorkspace> g_static;

int run_host_static(int dtype, const void* re_in, const void* im_in, void* re_out, void* im_out,
                    int n, int64_t batch, int normalize, cudaStream_t stream) {
  // every argument error (a vector too large for the static buffer included) comes
  // back before any CUDA call
  HostPlan hp;
  int st = validate_host(dtype, re_in, im_in, re_out, im_out, n, batch, normalize,
                         kStaticWorkspaceBytes, hp);
  if (st != FWT_OK || batch == 0) return st;
  std::lock_guard<std::mutex> lock(g_static_mu);
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess && (int)g_static.size() <= dev) g_static.resize(dev + 1);
  StaticWorkspace* sw = err == cudaSuccess ? &g_static[dev] : nullptr;
  if (err == cudaSuccess && !sw->ptr) {  // first call on this device
    err = cudaGetSymbolAddress(&sw->ptr, g_static_workspace);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&sw->done, cudaEventDisableTiming);
    if (err != cudaSuccess) sw->ptr = nullptr;
  }
  if (err == cudaSuccess && sw->used) err = cudaStreamWaitEvent(stream, sw->done, 0);
  if (err != cudaSuccess) {
    set_last_cuda_error((int)err);
    return FWT_ERR_CUDA;
  }
  bool started = false;
  st = enqueue_host(dtype, re_in, im_in, re_out, im_out, n, batch, normalize, sw->ptr, hp, stream,
                    started);
  // Once anything was enqueued, the next call must wait for it even when this one
  // failed part-way: the failed call's copies were joined back into `stream`.
  if (started) {
    err = cudaEventRecord(sw->done, stream);
    if (err == cudaSuccess) {
      sw->used = true;
    } else if (st == FWT_OK) {
      set_last_cuda_error((int)err);
      st = FWT_ERR_CUDA;
    }
  }
  return st;
}

}  // namespace
}  // namespace fwt

extern "C" {

size_t fwt_host_static_workspace_bytes(void) { return fwt::kStaticWorkspaceBytes; }

int fwt_host_static_c32(const float* re_in, const float* im_in, float* re_out, float* im_out,
                        int n, int64_t batch, int normalize, fwt_stream_t stream) {
  return fwt::run_host_static(FWT_C32, re_in, im_in, re_out, im_out, n, batch, normalize,
                              (cudaStream_t)stream);
}

int fwt_host_static_c64(const double* re_in, const double* im_in, double* re_out,
                        double* im_out, int n, int64_t batch, int normalize,
                        fwt_stream_t stream) {
  return fwt::run_host_static(FWT_C64, re_in, im_in, re_out, im_out, n, batch, normalize,
                              (cudaStream_t)stream);
}

int fwt_host_static_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out,
                        int32_t* im_out, int n, int64_t batch, int normalize,
                        fwt_stream_t stream) {
  return fwt::run_host_static(FWT_I32, re_in, im_in, re_out, im_out, n, batch, normalize,
                              (cudaStream_t)stream);
}

}  // extern "C"
