/*
 * fwt.h -- batched Walsh-Hadamard transform on GB300 (sm_103a), C ABI.
 *
 * Operation (every entry point below):
 *
 *     y[k] = s * sum_{i=0}^{2^n - 1} (-1)^{popc(k & i)} x[i],   k = 0 .. 2^n - 1
 *
 * applied independently to each of `batch` vectors of 2^n amplitudes.  The sign
 * rule is the natural-order (Sylvester) Hadamard matrix stated in
 * "[QDP] [feature] Pr4 kronecker fwt", section "How" (the on-the-fly Hadamard
 * value popc(k & i) of the naive GEMM placeholder).  s = 2^{-n/2} when
 * `normalize` is non-zero, else 1.  The complex state is held as split real and
 * imaginary arrays (the d_temp_real / d_temp_imag split of the same page); H is
 * real, so each part is transformed on its own.
 *
 * Layout: batch-major and contiguous.  Vector b of each array occupies elements
 * [b * 2^n, (b + 1) * 2^n).  Each array holds batch * 2^n elements.
 *
 * Memory and ownership: every pointer is a DEVICE pointer owned by the caller
 * (the fwt_host_* entry points alone take host arrays and a device workspace).
 * The library allocates no memory and never synchronises with the host: the
 * work is enqueued on `stream` (NULL = the legacy default
 * stream of the current device) and the call returns at once.  Results are
 * valid after the caller synchronises with `stream`.  Pointers must be 16-byte
 * aligned (every cudaMalloc / PyTorch allocation is).
 *
 * In-place: re_out == re_in and/or im_out == im_in (exactly) is allowed.  Any
 * other overlap between an output array and any array is rejected.
 *
 * Errors are returned synchronously.  Argument errors (INVALID_ARG, MISALIGNED,
 * UNSUPPORTED) are detected before anything is launched, so such a call has
 * enqueued no work.  FWT_ERR_CUDA means a CUDA call or launch failed;
 * fwt_last_cuda_error() returns its cudaError_t.  A multi-pass transform may
 * then have enqueued its earlier passes, and the output arrays are undefined.
 * Faults that happen later on the device surface at the caller's
 * synchronisation with `stream`.
 *
 * Thread safety: calls may be made from several host threads and devices; the
 * per-device set-up (kernel attributes, and the table of the fp64 phase copied to
 * the device) is done once under a lock, by the first call on each device: make that
 * call before capturing transforms into a CUDA graph.  Afterwards the entry points
 * enqueue only stream work.
 */
#ifndef FWT_GB300_H
#define FWT_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *); NULL is the default stream. */
typedef struct CUstream_st* fwt_stream_t;

enum fwt_status {
  FWT_OK = 0,
  FWT_ERR_INVALID_ARG = 1, /* bad n / batch / null pointer / overlapping arrays */
  FWT_ERR_MISALIGNED = 2,  /* a pointer is not 16-byte aligned */
  FWT_ERR_UNSUPPORTED = 3, /* e.g. normalize with int32, or a plan the build lacks */
  FWT_ERR_CUDA = 4,        /* a CUDA call failed; see fwt_last_cuda_error() */
  FWT_ERR_TIMEOUT = 5      /* a bounded device wait gave up (see fwt_device_status) */
};

enum fwt_dtype { FWT_C32 = 0, FWT_C64 = 1, FWT_I32 = 2 };

/*
 * Complex fp32, split re/im.  0 <= n <= 30, batch >= 0 (batch == 0 is a no-op
 * and accepts NULL pointers).  All four pointers must be non-NULL for batch > 0.
 * Arithmetic is fp32 add/sub; the relative L2 error per vector is within
 * n * 2^-24 of the exact transform of the input.
 */
int fwt_batched_c32(const float* re_in, const float* im_in, float* re_out, float* im_out,
                    int n, int64_t batch, int normalize, fwt_stream_t stream);

/*
 * Complex fp64, split re/im.  Same arguments as fwt_batched_c32.  The butterflies
 * run exactly in 64-bit fixed point on the integer units (one shared binary
 * exponent per on-chip tile), with a single rounding back to fp64 per pass; the
 * relative L2 error per vector stays below 1e-12 for finite input.  A tile that
 * holds an Inf or NaN is transformed in plain IEEE fp64 instead, so Inf/NaN
 * propagate as in IEEE arithmetic.
 */
int fwt_batched_c64(const double* re_in, const double* im_in, double* re_out, double* im_out,
                    int n, int64_t batch, int normalize, fwt_stream_t stream);

/*
 * Exact int32 variant: add/sub modulo 2^32 (two's complement wrap), bit-exact.
 * normalize must be 0 (2^{-n/2} is not an integer): FWT_ERR_UNSUPPORTED otherwise.
 * Real-only input: pass im_in == im_out == NULL (both, or neither).
 */
int fwt_batched_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out,
                    int32_t* im_out, int n, int64_t batch, int normalize, fwt_stream_t stream);

/*
 * Transform on a range of index bits (qubits): y = (I (x) H_nbits (x) I_{2^lo}) x
 * for each vector, i.e. the butterfly stages of index bits [lo, lo + nbits) only,
 * scaled by 2^{-nbits/2} when normalising.  lo = 0, nbits = n is the whole
 * transform; disjoint ranges compose, so a caller can apply the factors of a
 * Kronecker split one at a time ("[QDP] [feature] Pr4 kronecker fwt",
 * deliverables: (H_{n1} (x) I) and (I (x) H_{n2})).  0 <= lo, 0 <= nbits,
 * lo + nbits <= n <= 30; other arguments, layout, in-place rules and errors as
 * for fwt_batched_*.  Bits below 2^15 (2^14 for fp64) are handled in contiguous
 * tiles, higher bits by strided column tiles, each pass one read and one write.
 */
int fwt_bits_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream);
int fwt_bits_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream);
int fwt_bits_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, int lo, int nbits, int normalize, fwt_stream_t stream);

/*
 * Transform on an arbitrary set of index bits (qubits): bit i of `mask` set means
 * the butterfly stage of index bit i runs, i.e. y = (H or I per bit, Kronecker
 * product) x, scaled by 2^{-popcount(mask)/2} when normalising ("[QDP] [feature]
 * Pr4 kronecker fwt", deliverables: the factors (H_{n1} (x) I) and (I (x) H_{n2}) of
 * the two-stage form, generalised to any subset of the factors H_2 of H_n).  mask
 * must be below 2^n (else FWT_ERR_INVALID_ARG); 0 copies (scaled by 1).  A
 * contiguous mask is the same call as fwt_bits_*.  Otherwise the set bits below
 * 2^15 (2^14 for fp64) run in one pass over contiguous tiles with run-time
 * butterfly masks, and each contiguous run above in strided column passes.  Other
 * arguments, layout, in-place rules and errors as for fwt_batched_*.
 */
int fwt_mask_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream);
int fwt_mask_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream);
int fwt_mask_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, uint32_t mask, int normalize, fwt_stream_t stream);

/*
 * Diagonal phase, then transform (the IQP-encoding step: the state is multiplied
 * by a diagonal of phases before the Hadamard layer; "[QDP] [feature] Pr4
 * kronecker fwt", IQP shared-mem fused path):
 *
 *     y = s * H (e^{i theta} . x),   theta[b * theta_stride + i] for vector b,
 *
 * complex fp32, split re/im.  The pages do not give the angle function, so the
 * angles are an input: a DEVICE array of fp32 radians, theta_stride elements
 * between vectors (0: one row of 2^n angles shared by the batch; 2^n: one row per
 * vector).  theta must be 16-byte aligned, theta_stride a multiple of 4 when
 * n >= 2, and the angle array must not overlap the outputs (a theta_stride whose
 * angle extent, (batch - 1) * theta_stride + 2^n elements, does not fit in 64-bit
 * byte offsets is FWT_ERR_INVALID_ARG).  Phases come from
 * sincosf; the rotation is fused into the first pass (one read of x and theta,
 * one write), later passes as in fwt_batched_c32.  The relative L2 error per
 * vector stays within 2e-6 of the exact result.  Other arguments, in-place rules
 * and errors as fwt_batched_c32 (both parts are required).
 */
int fwt_phase_c32(const float* re_in, const float* im_in, const float* theta,
                  int64_t theta_stride, float* re_out, float* im_out, int n, int64_t batch,
                  int normalize, fwt_stream_t stream);

/*
 * The same for complex fp64 with fp64 angles: theta is a DEVICE array of doubles,
 * 16-byte aligned, theta_stride even when n >= 1.  The phase is applied element by
 * element into the outputs, and the fp64 transform then runs in place on them.  The
 * sine and cosine are evaluated in 64-bit integer arithmetic (GB300's fp64 unit is
 * slow): the angle reduced to a 64-bit fraction of a turn with 1/(2 pi) held to 128
 * bits, a 1024-entry table of cos/sin and short Taylor series for the remainder,
 * the rotation in fixed point with one rounding back to fp64; each rotated element
 * is within about 1e-16 of the exact rotation of its angle, relative to its
 * magnitude, for |theta| < 2^40.  Elements with an Inf or NaN, and angles of 2^40
 * and more, use the double-precision sincos instead.  Other arguments and errors as
 * fwt_phase_c32.
 */
int fwt_phase_c64(const double* re_in, const double* im_in, const double* theta,
                  int64_t theta_stride, double* re_out, double* im_out, int n, int64_t batch,
                  int normalize, fwt_stream_t stream);

/*
 * Host-buffer transform: the same operation as fwt_batched_* on arrays in HOST
 * memory, copied to the device, transformed and copied back.  (The pages describe
 * the on-device transform only; this is the end-to-end form of it.)
 *
 * re_in, im_in, re_out, im_out: HOST pointers, layout as above (im_in == im_out
 * == NULL allowed for int32 only).  Page-locked (pinned) host memory lets the
 * copies run asynchronously and overlap; pageable memory works, with copies that
 * serialise.  Each output may coincide exactly with its own input; any other
 * overlap is rejected.
 *
 * workspace: DEVICE memory of workspace_bytes bytes, owned by the caller, 16-byte
 * aligned; the library allocates nothing.  The batch is cut into chunks of whole
 * vectors and the workspace holds up to three chunks at a time: the host-to-device
 * copy of one chunk, the in-place transform of the previous one (on `stream`) and
 * the device-to-host copy of the one before run concurrently, the copies on two
 * streams the library creates once per device.  fwt_host_workspace_bytes() gives
 * the size that lets the pipeline run at full depth; a smaller workspace gives
 * smaller chunks or fewer slots, and one too small for a single vector is
 * FWT_ERR_INVALID_ARG.
 *
 * Asynchronous like the device entry points: the call returns once everything is
 * enqueued, and the outputs are complete when `stream` has reached the point of
 * the call (e.g. after cudaStreamSynchronize(stream)).  Work enqueued on `stream`
 * before the call completes before any copy starts.  The host buffers and the
 * workspace must stay untouched until then.  Calls are serialised per process
 * while they enqueue.  Errors as for fwt_batched_*; after FWT_ERR_CUDA earlier
 * chunks may have been enqueued and the outputs are undefined.
 */
int fwt_host_c32(const float* re_in, const float* im_in, float* re_out, float* im_out, int n,
                 int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream);
int fwt_host_c64(const double* re_in, const double* im_in, double* re_out, double* im_out, int n,
                 int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream);
int fwt_host_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out, int32_t* im_out,
                 int n, int64_t batch, int normalize, void* workspace, size_t workspace_bytes,
                 fwt_stream_t stream);

/*
 * Workspace bytes for fwt_host_* at full pipeline depth: three chunks of about
 * batch / 16 vectors (at least 32 MiB, at most the batch), both parts unless
 * with_im == 0 (int32 only).  0 for invalid arguments.
 */
size_t fwt_host_workspace_bytes(int dtype, int n, int64_t batch, int with_im);

/*
 * fwt_host_* without a caller workspace, for callers that cannot allocate device
 * memory: a plug-in or library running inside a host application that owns the
 * device memory (its own pool, or a fixed budget set at start-up) and forbids
 * stray cudaMalloc calls, or a latency-bound loop that cannot afford cudaMalloc's
 * implicit device synchronisation.  The pages have no counterpart of this entry
 * point: it is a convenience of the host-buffer path.
 *
 * The staging buffer is the library's own static device memory: a file-scope
 * __device__ array of fwt_host_static_workspace_bytes() bytes (512 MiB) that is
 * part of the module image, so nothing is allocated at run time (no cudaMalloc,
 * cudaFree or allocating library call).  Every device that loads the module holds
 * the array until the process exits: from the first call under CUDA's lazy module
 * loading (the default), from context creation under eager loading.
 *
 * The first call on a device does a one-time set-up with that device current: it
 * looks up the array's device address (cudaGetSymbolAddress) and creates an event.
 * Make that first call before any stream capture.  The address and the event are
 * kept for the life of the process: they, like the copy streams of fwt_host_*, do
 * not survive cudaDeviceReset or the destruction of the device's primary context.
 *
 * Same operation, arguments, layout, in-place rules, asynchrony and errors as
 * fwt_host_*.  Every argument error is returned before any CUDA call; in
 * particular a vector (both parts) larger than the static buffer is
 * FWT_ERR_INVALID_ARG.  Calls share the buffer, which keeps the last call's staged
 * data (every call overwrites what it reads before reading it).  Calls in one
 * process do not overlap on the GPU: each call makes `stream` wait until the
 * previous call (any stream, same device) has copied its last chunk out, also when
 * that call failed part-way.
 */
int fwt_host_static_c32(const float* re_in, const float* im_in, float* re_out, float* im_out,
                        int n, int64_t batch, int normalize, fwt_stream_t stream);
int fwt_host_static_c64(const double* re_in, const double* im_in, double* re_out,
                        double* im_out, int n, int64_t batch, int normalize,
                        fwt_stream_t stream);
int fwt_host_static_i32(const int32_t* re_in, const int32_t* im_in, int32_t* re_out,
                        int32_t* im_out, int n, int64_t batch, int normalize,
                        fwt_stream_t stream);
size_t fwt_host_static_workspace_bytes(void);

/* Static text for a status code (never NULL). */
const char* fwt_status_string(int status);

/* cudaError_t (as int) of the most recent FWT_ERR_CUDA on this host thread, else 0. */
int fwt_last_cuda_error(void);

/*
 * Number of HBM passes (one full read + write of the data each) the transform of
 * a 2^n vector of `dtype` takes with the current plan: 1 while a vector fits one
 * on-chip tile, 2 or 3 for the Kronecker split H_n = H_a (x) H_b (x) ...
 * ("[QDP] [feature] Pr4 kronecker fwt", section "Why": H_n = H_{n/2} (x) H_{n/2};
 * iThome "Day 18" FWT post, section "Kronecker block GEMM idea": H_N = H_a (x) H_b).
 * Returns -1 for an invalid n or dtype.
 */
int fwt_plan_passes(int n, int dtype);

/*
 * Writes the factor sizes of the plan for (n, dtype), lowest index bits first,
 * into bits[0 .. max_factors-1] and returns the number of factors (passes), or
 * -1 for invalid input.  The factors sum to n.
 */
int fwt_plan_factors(int n, int dtype, int* bits, int max_factors);

/*
 * Plan log: with the environment variable FWT_LOG set to anything but "" or "0"
 * (read once per process), every transform, bit-range, bit-mask and phase call
 * prints one line to stderr before it launches: the dtype, n, batch and each planned
 * pass (kind, transformed bits K, tile size, and for column passes the row stride,
 * segment width and mover).  Host-buffer calls print one line per chunk.
 */

/*
 * Tuning / testing: replace the plan for (n, dtype) by the given Kronecker
 * factors (low bits first; nfactors in 1..3; each factor must be supported by a
 * compiled tile shape, else FWT_ERR_UNSUPPORTED).  nfactors == 0 restores the
 * default plan.  Applies process-wide to calls issued after it returns.
 */
int fwt_set_plan(int n, int dtype, int nfactors, const int* bits);

/*
 * Tuning: bytes of contiguous columns (16, 32, 64 or 128) that each tile of a
 * column pass reads from every row it touches.  Wider segments make longer DRAM
 * bursts; narrower ones shrink the tile so that more CTAs share an SM, or let a
 * column factor grow.  16-byte tiles are always staged by TMA copies.  0 (the
 * default) chooses per plan: 64 bytes (fp32/int32) or 32 (fp64), and the measured
 * two-pass splits with narrower segments for large n (4-byte n = 26..28, fp64
 * n = 26); a plan set with fwt_set_plan gets the first width whose tiles cover its
 * factors.  Affects default plans and plans set afterwards for `dtype`.  Returns
 * FWT_OK or FWT_ERR_INVALID_ARG; fwt_get_column_bytes returns the setting (0 =
 * per plan, -1 for an invalid dtype).
 */
int fwt_set_column_bytes(int dtype, int bytes);
int fwt_get_column_bytes(int dtype);

/*
 * How column passes move their strided tiles: mode 2 stages every tile through
 * shared memory with TMA (cp.async.bulk.tensor) copies, 0 uses 16-byte vector
 * loads and stores, 1 (default) uses TMA for column factors of 10 or more bits
 * (tiles of 1024+ rows) and vector loads below, except in the measured default plans
 * that choose the mover per column factor (fp64 n = 15..22 and 26..30).  16-byte
 * column segments exist only as TMA tiles in every mode; an out-of-place call whose
 * first pass needs one copies its input to the output first.  Modes 1 and 2 also stage whole
 * fp64 row tiles with untiled bulk copies (cp.async.bulk); mode 0 loads them with
 * vector loads.  All modes give identical results.  Affects default plans and
 * plans set afterwards.  Returns FWT_OK or
 * FWT_ERR_INVALID_ARG; fwt_get_tma returns the mode.
 */
int fwt_set_tma(int mode);
int fwt_get_tma(void);

/*
 * One-pass cluster transform (fp32 / int32): a vector of 2^14 .. 2^18 elements is
 * spread over a thread-block cluster of 2 .. 16 CTAs; each CTA transforms the low
 * bits of its slice on chip, and the top bits are transformed across the cluster
 * through distributed shared memory, so the vector costs one HBM read and one
 * write instead of two of each (two Kronecker passes).  mode 1 (default): for
 * n = 15 .. 17 (where it measured at least as fast as the factor plans) when the
 * device can hold such a cluster; 2: for every n from 14 to 18; 0: never (factor plans
 * only).  fp64 uses CTA pairs for 2^14-element vectors (modes 1 and 2), as the
 * whole transform at n = 14 and as the 14-bit row pass of longer vectors: one
 * fixed-point exponent over the pair keeps the error bound only up to 2^14
 * elements.  Plans set with fwt_set_plan take precedence (a 14-bit fp64 row factor
 * still runs on pairs unless the mode is 0).  Returns FWT_OK or
 * FWT_ERR_INVALID_ARG; fwt_get_cluster returns the mode.
 */
int fwt_set_cluster(int mode);
int fwt_get_cluster(void);

/*
 * Launch overlap: mode 1 (default) launches pass kernels of up to 2048 CTAs with
 * programmatic stream serialisation, so one may be scheduled while the previous
 * kernel on the same stream is still finishing; each kernel waits
 * (griddepcontrol.wait) before its first global-memory access until that kernel has
 * completed and its writes are visible, so ordering on the stream is as without it.
 * It shortens back-to-back launches of small transforms (larger grids launch
 * plainly: there it measured neutral or slower).  Mode 0 launches every kernel
 * plainly.  Results are identical.  Returns FWT_OK or FWT_ERR_INVALID_ARG;
 * fwt_get_pdl returns the mode.
 */
int fwt_set_pdl(int mode);
int fwt_get_pdl(void);

/* Tuning: L2 sector promotion (0, 64, 128 (default) or 256 bytes) of the TMA
 * copies of column tiles.  Returns FWT_OK or FWT_ERR_INVALID_ARG. */
int fwt_set_tma_l2_promotion(int bytes);

/*
 * Device-side status: returns FWT_ERR_TIMEOUT if, since the last call, some kernel
 * gave up a bounded wait for a TMA copy (that tile was left unwritten), else
 * FWT_OK; clears the record.  Synchronises the device (it reads device memory).
 */
int fwt_device_status(void);

/*
 * Self-test of the bounded device wait: enqueues on `stream` one CTA that waits
 * on an mbarrier nobody arrives at (no copy targets it), so the wait gives up
 * after about one second and records a timeout; afterwards fwt_device_status()
 * returns FWT_ERR_TIMEOUT (and clears it).  Nothing is left in flight.  Returns
 * FWT_OK when enqueued.
 */
int fwt_selftest_bounded_wait(fwt_stream_t stream);

/*
 * L2 chunking of multi-pass transforms (tuning): when a plan has two or more
 * passes, the library runs all passes on one group of whole vectors before the
 * next group, so each intermediate is read back from L2 rather than DRAM.  A
 * group holds as many vectors as fit `bytes` (both parts in one launch when a
 * re/im pair fits, else one part at a time).  bytes = -1: half the L2 of the
 * current device; 0 (default): no chunking (one launch per pass over the batch).
 * Vectors larger than the budget are never chunked.  Process-wide; returns
 * FWT_OK or FWT_ERR_INVALID_ARG.  fwt_get_l2_chunk_bytes returns the setting.
 */
int fwt_set_l2_chunk_bytes(long long bytes);
long long fwt_get_l2_chunk_bytes(void);

/*
 * Per-pass tracing with caller-owned CUDA events (tracing without a profiler).
 * fwt_trace_events(events, capacity) arms tracing for the calling host thread:
 * every pass launched afterwards by this thread is bracketed by two
 * cudaEventRecord calls on the launch stream, into events[2i] and events[2i+1]
 * (events are cudaEvent_t handles created by the caller, with timing enabled),
 * until `capacity` events are used.  capacity == 0 disarms.  fwt_trace_count()
 * returns how many events have been recorded since arming.  The library creates,
 * destroys and synchronises nothing.  Returns FWT_OK or FWT_ERR_INVALID_ARG.
 */
int fwt_trace_events(void** events, int capacity);
int fwt_trace_count(void);

/*
 * Host-only self-check of every compiled tile shape: runs the kernels' index
 * maps on the CPU and verifies that each pass touches every element of its tile
 * exactly once, transforms every index bit of its factor exactly once, and that
 * every shared-memory access pattern is free of bank conflicts.  Returns 0 when
 * all shapes pass, else the number of failures (details to stderr).  Needs no GPU.
 */
int fwt_selfcheck(void);

#ifdef __cplusplus
}
#endif

#endif /* FWT_GB300_H */
