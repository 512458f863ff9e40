// specv_noalloc.cu -- a verify entry point that allocates no memory.
//
// Some callers cannot let a library allocate device memory while they run:
// code that owns the whole device allocator (a serving engine that carves all
// of HBM into its own pools up front), code running where an allocation
// would synchronise or fail (inside a latency-critical decode loop, or under
// a memory budget that is already fully committed), and callers that must
// guarantee the call never returns an out-of-memory error.  specv_verify
// allocates its small scratch workspace itself (once per stream, or per call
// while a graph is being captured); specv_verify_noalloc instead uses a fixed
// scratch array that is
// part of the library's device image (a file-scope __device__ array, created
// when the library's device code is loaded on a GPU and kept until the
// process exits).
//
// It runs the streaming cluster row kernel -- the same kernel, arithmetic and
// results as specv_verify gives when it plans that kernel -- with its
// per-position statistics and per-sequence arrival counters placed in that
// array.  Consequences for the caller:
//   - sizes are limited by the array: B*(K+1) <= kNoAllocMaxPositions and
//     B <= kNoAllocMaxSequences (larger calls return SPECV_ERR_INVALID_ARG and
//     launch nothing);
//   - every call on a device shares the one array: calls whose work overlaps
//     on that GPU (different streams, or several host threads) race on it and
//     must be serialised by the caller (e.g. one stream);
//   - the first call on a device looks up the array's device address (and
//     loads the library's kernels there); make that first call before any
//     CUDA graph capture.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "specv.h"
#include "specv_internal.h"

namespace {

constexpr int64_t kNoAllocMaxPositions = 49152;   // B*(K+1): 16 bytes each (768 KiB)
constexpr int64_t kNoAllocMaxSequences = 65536;   // B: 4 bytes each (256 KiB)
constexpr int64_t kStatsBytes = kNoAllocMaxPositions * 16;
constexpr int64_t kScratchBytes = kStatsBytes + kNoAllocMaxSequences * 4;  // 1 MiB
constexpr int kMaxDevices = 64;

// The scratch: statistics [B][K+1] (float4), then counters [B] (uint32).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Once per device, with that device current: the array's device address, the
// kernel attributes, and the SM count.
specv_status setup(int *dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    specv::note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SPECV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_lock);
  if (g_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      specv::note_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      (void)cudaGetLastError();
      return SPECV_ERR_CUDA;
    }
    int major = 0, cluster_ok = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      specv::note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_CUDA;
    }
    if (major < 10 || !cluster_ok) return SPECV_ERR_UNSUPPORTED;
    if ((e = specv::rows_prepare()) != cudaSuccess) {
      specv::note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_CUDA;
    }
    g_sms[dev] = sms;
    g_scratch_ptr[dev] = ptr;
  }
  *dev_out = dev;
  return SPECV_OK;
}

}  // namespace

extern "C" specv_status specv_verify_noalloc(const void *target_logits, const void *draft_logits,
                                             const int32_t *draft_tokens, const float *u_accept,
                                             const float *u_resample, const float *lambda,
                                             int64_t B, int32_t K, int32_t V, specv_dtype dtype,
                                             specv_mode mode, int32_t *out_tokens,
                                             int32_t *out_n_accepted, void *stream) {
  if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_resample || !lambda ||
      !out_tokens || !out_n_accepted)
    return SPECV_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || K > 4096 || V < 1) return SPECV_ERR_INVALID_ARG;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (mode != SPECV_PROB_MIX && mode != SPECV_LOGIT_MIX && mode != SPECV_GREEDY)
    return SPECV_ERR_INVALID_ARG;
  if (B > kNoAllocMaxSequences || B * (K + 1) > kNoAllocMaxPositions) return SPECV_ERR_INVALID_ARG;
  int dev = 0;
  specv_status st = setup(&dev);
  if (st != SPECV_OK) return st;

  const int bf16 = dtype == SPECV_BF16;
  const int elem = bf16 ? 2 : 4;
  const int vw = 16 / elem;
  const int64_t P = B * (K + 1);
  const int64_t G = (V + vw - 1) / vw;
  const int64_t row_bytes = (int64_t)V * elem;
  // cluster size: the streaming kernel's rule
  const int S = specv::stream_cluster_size(P, row_bytes, G, g_sms[dev]);

  unsigned char *scratch = static_cast<unsigned char *>(g_scratch_ptr[dev]);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  specv::RowArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.tokens = draft_tokens;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.lam = lambda;
  a.B = B;
  a.K = K;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_n = out_n_accepted;
  a.ws_stats = reinterpret_cast<float4 *>(scratch);
  a.ws_count = reinterpret_cast<unsigned *>(scratch + kStatsBytes);
  a.dbg_ptilde = nullptr;
  a.dbg_q = nullptr;
  a.dbg_lse = nullptr;
  a.groups_per_slice = (int)((G + S - 1) / S);
  a.num_groups = (int)G;
  // no room for the bonus rows' segment statistics: the sampler reads the bonus row again
  specv::rows_segments(a.groups_per_slice, &a.seg_tiles, &a.segs_per_slice);
  a.ws_seg = nullptr;
  a.defer_sampling = 0;  // one launch: the token draws stay in the statistics launch
  a.stats_cluster = S;
  a.stats_groups_per_slice = a.groups_per_slice;
  a.stats_seg_tiles = a.seg_tiles;
  a.stats_segs_per_slice = a.segs_per_slice;
  const bool aligned = ((uintptr_t)target_logits % 16 == 0) && ((uintptr_t)draft_logits % 16 == 0) &&
                       (row_bytes % 16 == 0);
  // the arrival counters must start at zero on every call (no allocation: a memset)
  cudaError_t e = cudaMemsetAsync(a.ws_count, 0, (size_t)B * sizeof(unsigned), s);
  if (e == cudaSuccess) e = specv::rows_launch(a, bf16, mode, aligned, S, P * S, s);
  if (e != cudaSuccess) {
    specv::note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}
