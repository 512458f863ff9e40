// specv_api.cu -- the C ABI of libspecv.so (declared in include/specv.h).
//
// Host-side work only: argument validation, the launch plan (which kernel,
// cluster size, grid), the per-call scratch workspace and the launches.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "specv.h"
#include "specv_internal.h"

namespace {
thread_local char g_last_cuda_error[256] = "";
}  // namespace

namespace specv {
void note_cuda_error(cudaError_t e) {
  std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
  g_last_cuda_error[sizeof(g_last_cuda_error) - 1] = '\0';
}
}  // namespace specv

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultSMs = 152;        // used by specv_plan when no device is visible
constexpr int64_t kDefaultL2 = 126LL * 1024 * 1024;
constexpr int kTileSmemBudget = 48 * 1024;
constexpr int kTmaTileStageBytes = 40 * 1024;  // target + draft rows of one staged tile, at most
// The tile size the planner aims for: two alternating tiles of 28 KiB let four
// CTAs share an SM (three with 40 KiB tiles).  Measured on the exactness
// workload (B = 10^6, K = 4, V = 32 fp32): 268.7 vs 280.9 us (probability),
// 234.4 vs 259.3 us (greedy), 316.0 vs 333.9 us (logit); smaller tiles cost
// more per-tile overhead than the extra CTA gains (24 KiB: 298.6 us).
constexpr int kTmaTileTargetBytes = 28 * 1024;
constexpr int kTileMaxV = 256;
constexpr int kTileMinSeqs = 4;
constexpr int kTileMaxSeqs = 64;
constexpr int32_t kMaxK = 4096;
// Resident row kernel: the staged slices of one CTA (target + draft) may use
// up to this much shared memory; the planner aims below kResidentTarget so
// that three CTAs fit an SM.
constexpr int kResidentMaxSmem = 200 * 1024;
constexpr int kResidentTarget = 96 * 1024;


struct DeviceState {
  bool ready = false;
  cudaError_t err = cudaSuccess;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

// Row-kernel scratch kept per (device, stream), in two parts: an array of
// per-sequence arrival counters, which starts at zero (cleared once when it is
// created) and which every completed launch leaves at zero again (the last
// cluster of each sequence resets its counter), and a data buffer for the
// position statistics or records, which needs no clearing.  Counters sit in a
// region of their own, so calls of any shape and kernel on one stream can
// share it.  A call therefore needs no allocation and no clearing step.
// A CUDA graph captured on a stream may hold the pointers, so a grown part's
// old buffer is not freed at once: it joins the entry's superseded list.
// Sizes double on growth, so the superseded buffers of an entry add up to
// less than its current ones.  specv_release_stream frees an entry (current
// and superseded buffers) when its owner says no graph will use them again.
struct Workspace {
  int dev;
  cudaStream_t stream;
  unsigned *count;
  int64_t count_len;
  void *data;
  size_t data_bytes;
  std::vector<void *> superseded;
};
std::vector<Workspace> g_ws;
constexpr size_t kWsMinBytes = 64 * 1024;

size_t grow_to(size_t need) {
  size_t sz = kWsMinBytes;
  while (sz < need) sz *= 2;
  return sz;
}

// The cached scratch of (dev, stream) with room for B counters and
// data_bytes, creating or growing it unless the stream is being captured.
// false if none can be used (the caller then takes stream-ordered memory).
bool cached_workspace(int dev, cudaStream_t stream, int64_t B, size_t data_bytes, unsigned **count,
                      void **data) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  Workspace *w = nullptr;
  for (Workspace &x : g_ws)
    if (x.dev == dev && x.stream == stream) w = &x;
  if (w != nullptr && w->count_len >= B && w->data_bytes >= data_bytes) {
    *count = w->count;
    *data = w->data;
    return true;
  }
  if (cap != cudaStreamCaptureStatusNone) return false;  // no allocation while capturing
  if (w == nullptr) {
    g_ws.push_back(Workspace{dev, stream, nullptr, 0, nullptr, 0, {}});
    w = &g_ws.back();
  }
  // grow a part by replacing it (the old part is kept: a graph may use it)
  if (w->count_len < B) {
    const size_t sz = grow_to((size_t)B * sizeof(unsigned));
    void *ptr = nullptr;
    if (cudaMalloc(&ptr, sz) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (cudaMemsetAsync(ptr, 0, sz, stream) != cudaSuccess) {
      (void)cudaGetLastError();
      (void)cudaFree(ptr);
      return false;
    }
    if (w->count != nullptr) w->superseded.push_back(w->count);
    w->count = static_cast<unsigned *>(ptr);
    w->count_len = (int64_t)(sz / sizeof(unsigned));
  }
  if (w->data_bytes < data_bytes) {
    const size_t sz = grow_to(data_bytes);
    void *ptr = nullptr;
    if (cudaMalloc(&ptr, sz) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (w->data != nullptr) w->superseded.push_back(w->data);
    w->data = ptr;
    w->data_bytes = sz;
  }
  *count = w->count;
  *data = w->data;
  return true;
}

using specv::note_cuda_error;

// One-time per-device set-up: opt the kernels into 16-CTA clusters and the
// tile kernel into its shared-memory size; read the SM count.
specv_status ensure_device(int *sms_out, int64_t *l2_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return SPECV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SPECV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState &st = g_dev[dev];
  if (!st.ready) {
    int major = 0, cluster_ok = 0, sms = 0, l2 = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    if (major < 10 || !cluster_ok) return SPECV_ERR_UNSUPPORTED;
    if ((e = specv::rows_prepare()) != cudaSuccess ||
        (e = specv::resident_prepare(kResidentMaxSmem)) != cudaSuccess ||
        (e = specv::tile_prepare(kTileSmemBudget)) != cudaSuccess ||
        (e = specv::tile_tma_prepare(2 * kTmaTileStageBytes + 16 * 1024)) != cudaSuccess ||
        (e = specv::alpha_prepare()) != cudaSuccess ||
        (e = specv::level_prepare()) != cudaSuccess ||
        (e = specv::tree_prepare()) != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    st.sms = sms;
    if (l2 > 0) st.l2 = l2;
    st.ready = true;
  }
  if (sms_out) *sms_out = st.sms;
  if (l2_out) *l2_out = st.l2;
  return SPECV_OK;
}

struct Plan {
  int kernel;            // 0 tile, 1 streaming row kernel, 2 resident row kernel, 3 TMA tile,
                         // 4 sequence-cluster row kernel
  int cluster;           // CTAs per cluster (row kernels)
  int64_t ctas;          // CTAs of the row kernels (tile kernel: tiles)
  int64_t ws_bytes;      // scratch bytes
  int tile_seqs;
  int smem_t, smem_d, smem_total;
  int groups_per_slice, num_groups;
  int seg_tiles, segs_per_slice;  // sampler segments of the streaming row kernel
  int res_smem;          // dynamic shared memory of the resident kernel
  int split;             // streaming kernel: 1 = token draws in a second launch (rows_sample)
  int sample_cluster;    // its cluster size
  int sample_gps, sample_seg_tiles, sample_segs;  // its slice and segment geometry
  int early_exit;        // streaming kernel: positions after a published rejection skip their rows
  int64_t counters;      // arrival counters in the scratch
};

int64_t round16(int64_t x) { return (x + 15) / 16 * 16; }

bool sizes_ok(int64_t B, int32_t K, int32_t V, int dtype, int mode) {
  if (B < 1 || K < 1 || K > kMaxK || V < 1) return false;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return false;
  if (mode != SPECV_PROB_MIX && mode != SPECV_LOGIT_MIX && mode != SPECV_GREEDY) return false;
  const int64_t lim = (int64_t)1 << 62;
  if (B > lim / (K + 1) || B * (K + 1) > lim / V) return false;
  return true;
}

int cluster_from_env() {
  const char *s = std::getenv("SPECV_CLUSTER_SIZE");
  if (!s || !*s) return 0;
  const int v = std::atoi(s);
  return (v >= 1 && v <= specv::kMaxCluster) ? v : 0;
}

// Early exit (the pages' loop stops at the first rejection): on grids of more
// than two waves the streaming kernels run position-major, every position
// publishes its own rejection, and a position after a published rejection
// reads none of its rows.  On grids of one or two waves every position streams
// at the same time, so none would be skipped.  SPECV_EARLY_EXIT=0 reads every
// row (tests, measurements).
bool early_exit_from_env() {
  const char *s = std::getenv("SPECV_EARLY_EXIT");
  return !(s && s[0] == '0');
}

// SPECV_SAMPLE_SPLIT=0/1 forces the streaming kernel's token draws into the
// statistics launch or into a second launch (tuning and tests); -1: the plan.
int split_from_env() {
  const char *s = std::getenv("SPECV_SAMPLE_SPLIT");
  if (!s || !*s) return -1;
  return s[0] == '1' ? 1 : (s[0] == '0' ? 0 : -1);
}

// "stream" or "resident" forces a row-kernel variant (tests of both kernels
// on one shape).
int variant_from_env() {
  const char *s = std::getenv("SPECV_ROWS_VARIANT");
  if (!s) return 0;
  if (std::strcmp(s, "stream") == 0) return 1;
  if (std::strcmp(s, "resident") == 0) return 2;
  return 0;
}

// The launch plan.
//  - Short rows whose whole sequences fit a shared-memory tile: tile kernel.
//  - Row kernels: the streaming cluster size is the smallest power of two
//    (<= 16) that gives the grid >= 4 CTAs per SM and each CTA <= 512 KiB of
//    (target + draft) slice, without going under 4 KiB of a row per CTA.
//  - The resident row kernel (16-byte aligned rows, slice in shared memory)
//    pays a fixed latency per CTA that only a single wave of clusters hides,
//    so it is chosen when its grid (smallest cluster size whose slice fits
//    96 KiB, doubled while the grid has < 4 CTAs per SM) stays within 2 CTAs
//    per SM; otherwise the streaming row kernel runs.
//  SPECV_CLUSTER_SIZE and SPECV_ROWS_VARIANT override the choices.
specv_status make_plan(int64_t B, int32_t K, int32_t V, int dtype, int mode, int sms, int64_t l2,
                       bool aligned, Plan *p, bool allow_tma = true) {
  const int elem = dtype == SPECV_BF16 ? 2 : 4;
  std::memset(p, 0, sizeof(*p));
  const bool greedy = mode == SPECV_GREEDY;
  const int64_t seq_bytes = (int64_t)(2 * K + 1) * V * elem + (int64_t)(K + 1) * 16;
  const int64_t data_bytes0 = (int64_t)(2 * K + 1) * V * elem;
  const bool tma0 = allow_tma && aligned && ((int64_t)V * elem) % 16 == 0 &&
                    data_bytes0 <= kTmaTileStageBytes;
  // greedy runs in the TMA tile kernel or the streaming row kernel only
  if (V <= kTileMaxV && seq_bytes * kTileMinSeqs + 64 <= kTileSmemBudget && (!greedy || tma0)) {
    const int64_t data_bytes = data_bytes0;
    const bool tma = tma0;
    int ts;
    if (tma) {
      // two alternating tile buffers of about 28 KiB (40 KiB at most); one round of stage-A
      // row tasks (2K+1 per sequence) for the CTA's threads; at most one
      // stage-B lane group per sequence
      ts = (int)(kTmaTileTargetBytes / data_bytes);
      const int by_rows = specv::kTmaTileThreads / (2 * K + 1);
      if (ts > by_rows && by_rows >= 1) ts = by_rows;
      if (ts > specv::kTmaTileMaxSeqs) ts = specv::kTmaTileMaxSeqs;
      if (ts < 1) ts = 1;
    } else {
      ts = (int)((kTileSmemBudget - 64) / seq_bytes);
      if (ts > kTileMaxSeqs) ts = kTileMaxSeqs;
    }
    if (ts > B) ts = (int)B;
    p->kernel = tma ? 3 : 0;
    p->cluster = 1;
    p->tile_seqs = ts;
    p->smem_t = (int)round16((int64_t)ts * (K + 1) * V * elem);
    p->smem_d = (int)round16((int64_t)ts * K * V * elem);
    p->smem_total = tma ? 128 + 2 * (p->smem_t + p->smem_d) + ts * (K + 1) * 16
                        : p->smem_t + p->smem_d + ts * (K + 1) * 16;
    p->ctas = (B + ts - 1) / ts;  // tiles
    p->ws_bytes = 0;
    return SPECV_OK;
  }
  const int64_t P = B * (K + 1);
  const int vw = 16 / elem;
  const int64_t row_bytes = (int64_t)V * elem;
  const int64_t G = (V + vw - 1) / vw;
  const int env_S = cluster_from_env();
  const int env_var = variant_from_env();
  const int64_t waves_slots = 2 * 4LL * sms;  // two waves of 4 CTAs per SM
  if (greedy) {
    // greedy needs no sampling pass: the streaming row kernel, one read of every logit
    if (env_var == 2) return SPECV_ERR_UNSUPPORTED;
    int S = env_S;
    if (S == 0) S = specv::stream_cluster_size(P, row_bytes, G, sms);
    while (S > 1 && P * S > INT32_MAX) S /= 2;
    if (P * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
    p->kernel = 1;
    p->cluster = S;
    p->ctas = P * S;
    p->num_groups = (int)G;
    p->groups_per_slice = (int)((G + S - 1) / S);
    specv::rows_segments(p->groups_per_slice, &p->seg_tiles, &p->segs_per_slice);
    p->counters = B;
    p->ws_bytes = round16(P * 16) + round16(B * 4);
    if (P * S > waves_slots && early_exit_from_env()) {  // early exit: one word per sequence
      p->early_exit = 1;
      p->counters = 2 * B;
      p->ws_bytes += round16(B * 4);
    }
    return SPECV_OK;
  }
  const bool can_resident = allow_tma && aligned && (row_bytes % 16 == 0) && env_var != 1;
  auto slice_smem = [&](int S) { return 2 * ((G + S - 1) / S) * 16; };
  int S = 0;
  int kernel = 1;
  if (can_resident) {
    if (env_S) {
      if (slice_smem(env_S) <= kResidentMaxSmem) S = env_S;
    } else {
      for (int s = 1; s <= specv::kMaxCluster; s *= 2)
        if (slice_smem(s) <= kResidentTarget) {
          S = s;
          break;
        }
      if (S == 0 && slice_smem(specv::kMaxCluster) <= kResidentMaxSmem) S = specv::kMaxCluster;
      if (S)
        while (S < specv::kMaxCluster && P * S < 4LL * sms && row_bytes / (2 * S) >= 4096) S *= 2;
    }
    if (S && env_var != 2 && P * S > 2LL * sms) S = 0;  // several waves: streaming is faster
    if (S) kernel = 2;
  }
  if (kernel == 2 && P * S > INT32_MAX) kernel = 1;
  if (env_var == 2 && kernel != 2) return SPECV_ERR_UNSUPPORTED;
  if (kernel == 1) {
    S = env_S;
    if (S == 0) S = specv::stream_cluster_size(P, row_bytes, G, sms);
    while (S > 1 && P * S > INT32_MAX) S /= 2;
    if (P * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
  }
  p->kernel = kernel;
  p->cluster = S;
  p->ctas = P * S;
  p->num_groups = (int)G;
  p->groups_per_slice = (int)((G + S - 1) / S);
  p->counters = B;
  if (kernel == 2) {
    p->res_smem = (int)slice_smem(S);
    p->ws_bytes = round16(P * 8) + round16(B * 4);
  } else {
    // position statistics, then the bonus rows' segment statistics
    specv::rows_segments(p->groups_per_slice, &p->seg_tiles, &p->segs_per_slice);
    p->ws_bytes = round16(P * 16) + round16(B * S * (int64_t)p->segs_per_slice * 8) + round16(B * 4);
    // A grid of about one wave finishes every sequence at about the same time,
    // so the last clusters' token draws form a tail on a few CTAs each; then
    // the draws run as a second launch with a wider cluster per sequence
    // (about 48 KiB of the row pair per CTA, mostly still in L2).  Several
    // waves keep the draws in the statistics launch, overlapped with streaming.
    const int env_split = split_from_env();
    const bool one_wave = P * S <= waves_slots;
    // About one wave of few sequences: one cluster of 16 CTAs per sequence
    // streams all its positions, decides it and draws its token in a single
    // launch (no scratch, no second launch), when 16 CTAs per sequence fit
    // one wave of 4 CTAs per SM and the clusters fill at least two CTAs per
    // SM (measured on GB300 against the two-launch plan: 39.6 against 43.7 us
    // at B = 32, K = 5, V = 152064 bf16; 41.6 against 49.8 us at B = 24,
    // K = 6, V = 40001; but with more sequences on smaller clusters the
    // two-launch plan wins: 33.4 against 27.3 us at B = 40, K = 3, V = 32000
    // on clusters of 15).  Device memory only: a forced variant, cluster size
    // or draw split keeps the streaming kernel.
    if (one_wave && allow_tma && env_split < 0 && env_var == 0 && env_S == 0) {
      const int64_t sq = specv::kMaxCluster;
      if (B * sq <= 4LL * sms && B * sq >= 2LL * sms && K + 1 <= specv::kSeqMaxPositions &&
          row_bytes / sq >= 4096) {
        p->kernel = 4;
        p->cluster = (int)sq;
        p->ctas = B * sq;
        p->groups_per_slice = (int)((G + sq - 1) / sq);
        specv::rows_segments(p->groups_per_slice, &p->seg_tiles, &p->segs_per_slice);
        p->counters = 0;
        p->ws_bytes = 0;
        return SPECV_OK;
      }
    }
    p->split = env_split >= 0 ? env_split : (one_wave ? 1 : 0);
    if (p->split) {
      int64_t s2 = (2 * row_bytes + 48 * 1024 - 1) / (48 * 1024);
      if (s2 < 1) s2 = 1;
      if (s2 > specv::kMaxCluster) s2 = specv::kMaxCluster;
      while (s2 > 1 && B * s2 > INT32_MAX) --s2;
      p->sample_cluster = (int)s2;
      p->sample_gps = (int)((G + s2 - 1) / s2);
      specv::rows_segments(p->sample_gps, &p->sample_seg_tiles, &p->sample_segs);
    }
    // Early exit: the grid runs position-major and a position skips its rows
    // when an earlier position of its sequence has published a rejection; one
    // more word per sequence in the counter region (zero at entry, left zero).
    if (!p->split && early_exit_from_env()) {
      p->early_exit = 1;
      p->counters = 2 * B;
      p->ws_bytes += round16(B * 4);
    }
  }
  return SPECV_OK;
}

specv_status run(const void *target, const void *draft, const int32_t *tokens, const float *ua,
                 const float *ur, const float *lam, int64_t B, int32_t K, int32_t V,
                 specv_dtype dtype, specv_mode mode, int32_t *out_tokens, int32_t *out_n,
                 float *dbg_ptilde, float *dbg_q, float *dbg_lse, void *stream_ptr,
                 bool allow_tma = true, void *mirror_t = nullptr, void *mirror_d = nullptr) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status s = ensure_device(&sms, &l2);
  if (s != SPECV_OK) return s;
  const int bf16 = dtype == SPECV_BF16;
  const int elem = bf16 ? 2 : 4;
  const bool aligned = ((uintptr_t)target % 16 == 0) && ((uintptr_t)draft % 16 == 0) &&
                       ((int64_t)V * elem % 16 == 0);
  Plan p;
  if ((s = make_plan(B, K, V, dtype, mode, sms, l2, aligned, &p, allow_tma)) != SPECV_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e;
  if (p.kernel == 0 || p.kernel == 3) {
    specv::TileArgs a;
    a.target = target;
    a.draft = draft;
    a.tokens = tokens;
    a.u_accept = ua;
    a.u_resample = ur;
    a.lam = lam;
    a.B = B;
    a.K = K;
    a.V = V;
    a.out_tokens = out_tokens;
    a.out_n = out_n;
    a.dbg_ptilde = dbg_ptilde;
    a.dbg_q = dbg_q;
    a.dbg_lse = dbg_lse;
    a.tile_seqs = p.tile_seqs;
    a.num_tiles = p.ctas;
    a.vec_copy = ((uintptr_t)target % 16 == 0) && ((uintptr_t)draft % 16 == 0) &&
                 ((int64_t)(K + 1) * V * elem % 16 == 0) && ((int64_t)K * V * elem % 16 == 0);
    a.smem_target_bytes = p.smem_t;
    a.smem_draft_bytes = p.smem_d;
    const int per_sm = p.kernel == 3 ? specv::tile_tma_blocks_per_sm(bf16, mode, p.smem_total)
                                     : specv::tile_blocks_per_sm(bf16, mode, p.smem_total);
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > p.ctas) grid = p.ctas;
    e = p.kernel == 3 ? specv::tile_tma_launch(a, bf16, mode, grid, p.smem_total, stream)
                      : specv::tile_launch(a, bf16, mode, grid, p.smem_total, stream);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    return SPECV_OK;
  }
  if (p.kernel == 4) {  // the sequence-cluster kernel: no scratch
    specv::RowArgs a;
    a.target = target;
    a.draft = draft;
    a.tokens = tokens;
    a.u_accept = ua;
    a.u_resample = ur;
    a.lam = lam;
    a.B = B;
    a.K = K;
    a.V = V;
    a.out_tokens = out_tokens;
    a.out_n = out_n;
    a.ws_stats = nullptr;
    a.ws_count = nullptr;
    a.dbg_ptilde = dbg_ptilde;
    a.dbg_q = dbg_q;
    a.dbg_lse = dbg_lse;
    a.groups_per_slice = p.groups_per_slice;
    a.num_groups = p.num_groups;
    a.seg_tiles = p.seg_tiles;
    a.segs_per_slice = p.segs_per_slice;
    a.ws_seg = nullptr;
    a.defer_sampling = 0;
    e = specv::rows_seq_launch(a, bf16, mode, aligned, p.cluster, stream);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    return SPECV_OK;
  }
  int dev = 0;
  (void)cudaGetDevice(&dev);
  // scratch: counters [B] then position data, from the stream's cache or,
  // failing that, stream-ordered memory for this call (counters cleared)
  const size_t data_bytes = (size_t)(p.ws_bytes - round16(p.counters * 4));
  unsigned *cnt = nullptr;
  void *wdata = nullptr;
  void *ws = nullptr;
  e = cudaSuccess;
  const bool per_call = !cached_workspace(dev, stream, p.counters, data_bytes, &cnt, &wdata);
  if (per_call) {
    e = cudaMallocAsync(&ws, (size_t)p.ws_bytes, stream);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_NO_MEMORY;
    }
    cnt = static_cast<unsigned *>(ws);
    wdata = static_cast<char *>(ws) + round16(p.counters * 4);
    e = cudaMemsetAsync(cnt, 0, (size_t)p.counters * sizeof(unsigned), stream);
  }
  if (p.kernel == 2) {
    specv::ResArgs r;
    r.target = target;
    r.draft = draft;
    r.tokens = tokens;
    r.u_accept = ua;
    r.u_resample = ur;
    r.lam = lam;
    r.B = B;
    r.K = K;
    r.V = V;
    r.out_tokens = out_tokens;
    r.out_n = out_n;
    r.rec = static_cast<int2 *>(wdata);
    r.count = cnt;
    r.dbg_ptilde = dbg_ptilde;
    r.dbg_q = dbg_q;
    r.dbg_lse = dbg_lse;
    r.groups_per_slice = p.groups_per_slice;
    r.num_groups = p.num_groups;
    if (e == cudaSuccess)
      e = specv::resident_launch(r, bf16, mode, p.cluster, p.ctas, p.res_smem, stream);
  } else {
    specv::RowArgs a;
    a.target = target;
    a.draft = draft;
    a.tokens = tokens;
    a.u_accept = ua;
    a.u_resample = ur;
    a.lam = lam;
    a.B = B;
    a.K = K;
    a.V = V;
    a.out_tokens = out_tokens;
    a.out_n = out_n;
    a.ws_stats = static_cast<float4 *>(wdata);
    a.ws_count = cnt;
    a.dbg_ptilde = dbg_ptilde;
    a.dbg_q = dbg_q;
    a.dbg_lse = dbg_lse;
    a.groups_per_slice = p.groups_per_slice;
    a.num_groups = p.num_groups;
    a.seg_tiles = p.seg_tiles;
    a.segs_per_slice = p.segs_per_slice;
    a.ws_seg = mode == SPECV_GREEDY ? nullptr  // no sampling, no segment statistics
                                    : reinterpret_cast<float2 *>(static_cast<char *>(wdata) +
                                                                 round16(B * (K + 1) * 16));
    a.defer_sampling = mode != SPECV_GREEDY && p.split;
    // early exit, except for the debug entry point (which reports every position)
    if (p.early_exit && dbg_ptilde == nullptr && dbg_lse == nullptr) {
      a.ws_reject = cnt + B;
      a.pos_major = 1;
    }
    if (aligned && mirror_t != nullptr && mirror_d != nullptr && mode != SPECV_GREEDY) {
      a.mirror_target = mirror_t;  // device copies of the rows streamed, for the token draws
      a.mirror_draft = mirror_d;
    }
    a.stats_cluster = p.cluster;
    a.stats_groups_per_slice = p.groups_per_slice;
    a.stats_seg_tiles = p.seg_tiles;
    a.stats_segs_per_slice = p.segs_per_slice;
    if (e == cudaSuccess)
      e = specv::rows_launch(a, bf16, mode, aligned, p.cluster, p.ctas, stream);
    if (e == cudaSuccess && a.defer_sampling) {
      specv::RowArgs a2 = a;
      a2.groups_per_slice = p.sample_gps;
      a2.seg_tiles = p.sample_seg_tiles;
      a2.segs_per_slice = p.sample_segs;
      e = specv::rows_sample_launch(a2, bf16, mode, aligned, p.sample_cluster,
                                    B * (int64_t)p.sample_cluster, stream);
    }
  }
  if (per_call) {
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

// ---------------------------------------------------------------------------
// Verify on host buffers.  Per (device, stream) the library keeps a copy
// stream, one event per chunk, and device staging memory for the inputs and
// outputs of one call.  The inputs of chunk c (whole sequences) are copied on
// the copy stream while the verify step of chunk c-1 runs on the caller's
// stream, so the host link and the kernels overlap; the link (not HBM) bounds
// such a call.  Staging grows by replacement after both streams have drained;
// a call never runs under stream capture, so no graph can hold staging memory.
constexpr int kHostMaxChunks = 64;
constexpr int kHostAutoMaxChunks = 16;
constexpr int64_t kHostChunkBytes = 64LL << 20;  // logit bytes per chunk (automatic choice)

struct HostPipe {
  int dev;
  cudaStream_t stream;
  cudaStream_t copy;
  cudaStream_t aux;        // the early-exit call's second decision stream
  cudaEvent_t start;
  cudaEvent_t ready[kHostMaxChunks];
  void *stage;
  size_t stage_bytes;
  unsigned char *h_alive;  // page-locked: the early-exit call's per-sequence flags
  size_t h_alive_bytes;
};
std::vector<HostPipe *> g_pipes;  // never freed while the process runs

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The pipe of (dev, stream) with at least `need` bytes of staging memory.
specv_status host_pipe(int dev, cudaStream_t stream, size_t need, HostPipe **out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  HostPipe *hp = nullptr;
  for (HostPipe *x : g_pipes)
    if (x->dev == dev && x->stream == stream) hp = x;
  cudaError_t e = cudaSuccess;
  if (hp == nullptr) {
    hp = new HostPipe{};
    hp->dev = dev;
    hp->stream = stream;
    e = cudaStreamCreateWithFlags(&hp->copy, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->aux, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming);
    for (int c = 0; c < kHostMaxChunks && e == cudaSuccess; ++c)
      e = cudaEventCreateWithFlags(&hp->ready[c], cudaEventDisableTiming);
    if (e != cudaSuccess) {  // a partly built pipe is leaked, not reused
      note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_CUDA;
    }
    g_pipes.push_back(hp);
  }
  if (hp->stage_bytes < need) {
    // earlier calls on this pipe may still read or write the old staging
    e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(hp->copy);
    if (e == cudaSuccess) e = cudaStreamSynchronize(hp->aux);
    if (e == cudaSuccess && hp->stage != nullptr) e = cudaFree(hp->stage);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_CUDA;
    }
    hp->stage = nullptr;
    hp->stage_bytes = 0;
    const size_t sz = grow_to(need);
    if (cudaMalloc(&hp->stage, sz) != cudaSuccess) {
      (void)cudaGetLastError();
      hp->stage = nullptr;
      return SPECV_ERR_NO_MEMORY;
    }
    hp->stage_bytes = sz;
  }
  *out = hp;
  return SPECV_OK;
}

specv_status verify_host(const void *target, const void *draft, const int32_t *tokens,
                         const float *ua, const float *ur, const float *lam, int64_t B, int32_t K,
                         int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                         int32_t *out_n, int32_t chunks, void *stream_ptr) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode) || chunks < 0 || chunks > kHostMaxChunks)
    return SPECV_ERR_INVALID_ARG;
  const size_t elem = dtype == SPECV_BF16 ? 2 : 4;
  // staging larger than any device's memory is refused before the products overflow
  if ((uint64_t)B * (uint64_t)(2 * K + 1) > ((uint64_t)1 << 50) / elem / (uint64_t)V)
    return SPECV_ERR_NO_MEMORY;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status s = ensure_device(&sms, &l2);
  if (s != SPECV_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return SPECV_ERR_UNSUPPORTED;
  int dev = 0;
  (void)cudaGetDevice(&dev);

  // staging layout: target, draft, tokens, u_accept, u_resample, lambda,
  // out_tokens, out_n (each region 256-byte aligned)
  const size_t row_bytes = (size_t)V * elem;
  const size_t t_bytes = (size_t)B * (K + 1) * row_bytes, d_bytes = (size_t)B * K * row_bytes;
  const size_t bk4 = (size_t)B * K * 4, b4 = (size_t)B * 4, bk14 = (size_t)B * (K + 1) * 4;
  const size_t o_d = round256(t_bytes), o_tok = o_d + round256(d_bytes);
  const size_t o_ua = o_tok + round256(bk4), o_ur = o_ua + round256(bk4);
  const size_t o_lam = o_ur + round256(b4), o_ot = o_lam + round256(b4);
  const size_t o_on = o_ot + round256(bk14), need = o_on + round256(b4);
  HostPipe *hp = nullptr;
  if ((s = host_pipe(dev, stream, need, &hp)) != SPECV_OK) return s;
  char *st = static_cast<char *>(hp->stage);

  int64_t nc = chunks;
  if (nc == 0) {
    nc = (int64_t)((t_bytes + d_bytes + kHostChunkBytes - 1) / kHostChunkBytes);
    nc = nc < 1 ? 1 : (nc > kHostAutoMaxChunks ? kHostAutoMaxChunks : nc);
  }
  if (nc > B) nc = B;
  auto chunk_lo = [&](int64_t c) { return c * (B / nc) + (c < B % nc ? c : B % nc); };

  // copies: after the caller's earlier work on `stream` (which may still read
  // the staging), the per-sequence arrays first, then the logits chunk by chunk
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  e = cudaEventRecord(hp->start, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->copy, hp->start, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_tok, tokens, bk4, h2d, hp->copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_ua, ua, bk4, h2d, hp->copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_ur, ur, b4, h2d, hp->copy);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_lam, lam, b4, h2d, hp->copy);
  for (int64_t c = 0; c < nc && e == cudaSuccess; ++c) {
    const int64_t b0 = chunk_lo(c), b1 = chunk_lo(c + 1);
    const size_t ot = (size_t)b0 * (K + 1) * row_bytes, od = (size_t)b0 * K * row_bytes;
    e = cudaMemcpyAsync(st + ot, static_cast<const char *>(target) + ot,
                        (size_t)(b1 - b0) * (K + 1) * row_bytes, h2d, hp->copy);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(st + o_d + od, static_cast<const char *>(draft) + od,
                          (size_t)(b1 - b0) * K * row_bytes, h2d, hp->copy);
    if (e == cudaSuccess) e = cudaEventRecord(hp->ready[c], hp->copy);
  }
  if (e != cudaSuccess) {  // nothing of this call has been launched on `stream`
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  // the verify step of each chunk, once its inputs are in
  for (int64_t c = 0; c < nc && s == SPECV_OK; ++c) {
    const int64_t b0 = chunk_lo(c), b1 = chunk_lo(c + 1);
    e = cudaStreamWaitEvent(stream, hp->ready[c], 0);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      s = SPECV_ERR_CUDA;
      break;
    }
    s = run(st + (size_t)b0 * (K + 1) * row_bytes, st + o_d + (size_t)b0 * K * row_bytes,
            reinterpret_cast<const int32_t *>(st + o_tok) + b0 * K,
            reinterpret_cast<const float *>(st + o_ua) + b0 * K,
            reinterpret_cast<const float *>(st + o_ur) + b0,
            reinterpret_cast<const float *>(st + o_lam) + b0, b1 - b0, K, V, dtype, mode,
            reinterpret_cast<int32_t *>(st + o_ot) + b0 * (K + 1),
            reinterpret_cast<int32_t *>(st + o_on) + b0, nullptr, nullptr, nullptr, stream);
  }
  if (s != SPECV_OK) {
    // join the copy stream so that the caller's stream covers every copy issued
    (void)cudaStreamWaitEvent(stream, hp->ready[nc - 1], 0);
    (void)cudaGetLastError();
    return s;
  }
  e = cudaMemcpyAsync(out_tokens, st + o_ot, bk14, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_n, st + o_on, b4, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

// ---------------------------------------------------------------------------
// Verify on host buffers that the device can read in place: the kernels load
// the rows they reach straight from host memory over the host link, so only
// those rows cross it (early exit skips the rest) and nothing waits for a
// copy to finish.  The host link is about 30 times slower than HBM, so the
// kernels spend most of the time waiting on it; the kernels that stage rows
// with bulk copies (the resident and TMA tile kernels) are not planned, the
// register-load kernels are.
//
// A host pointer qualifies when the runtime reports it page-locked and
// mapped (cudaHostAlloc, cudaHostRegister: its device address is used), or
// when it is ordinary host memory and the device reads pageable memory
// (cudaDevAttrPageableMemoryAccess, e.g. over a coherent CPU-GPU link).
bool device_address(const void *p, bool pageable_ok, const void **out) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = p;
    return true;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    // the same offset from the allocation's device address
    *out = static_cast<const char *>(at.devicePointer) +
           (static_cast<const char *>(p) - static_cast<const char *>(at.hostPointer));
    return true;
  }
  if (at.type == cudaMemoryTypeUnregistered && pageable_ok) {
    *out = p;
    return true;
  }
  return false;
}

specv_status verify_host_direct(const void *target, const void *draft, const int32_t *tokens,
                                const float *ua, const float *ur, const float *lam, int64_t B,
                                int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                int32_t *out_tokens, int32_t *out_n, void *stream_ptr) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status s = ensure_device(&sms, &l2);
  if (s != SPECV_OK) return s;
  int dev = 0, pageable = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  const void *in[6] = {target, draft, tokens, ua, ur, lam};
  const void *dv[6];
  for (int k = 0; k < 6; ++k)
    if (!device_address(in[k], pageable != 0, &dv[k])) return SPECV_ERR_UNSUPPORTED;
  const void *dot = nullptr, *don = nullptr;
  if (!device_address(out_tokens, pageable != 0, &dot) ||
      !device_address(out_n, pageable != 0, &don))
    return SPECV_ERR_UNSUPPORTED;
  // Device copies of the rows as they stream (the streaming kernel's token
  // draws read the rejected pair a second time, from HBM instead of across
  // the link): the pipe's staging memory, laid out like the inputs.
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(stream, &cap)) != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return SPECV_ERR_UNSUPPORTED;  // staging may grow
  const size_t elem = dtype == SPECV_BF16 ? 2 : 4;
  if ((uint64_t)B * (uint64_t)(2 * K + 1) > ((uint64_t)1 << 50) / elem / (uint64_t)V)
    return SPECV_ERR_NO_MEMORY;
  const size_t t_bytes = (size_t)B * (K + 1) * V * elem, d_bytes = (size_t)B * K * V * elem;
  HostPipe *hp = nullptr;
  if ((s = host_pipe(dev, stream, round256(t_bytes) + round256(d_bytes), &hp)) != SPECV_OK) return s;
  char *mir = static_cast<char *>(hp->stage);
  return run(dv[0], dv[1], static_cast<const int32_t *>(dv[2]), static_cast<const float *>(dv[3]),
             static_cast<const float *>(dv[4]), static_cast<const float *>(dv[5]), B, K, V, dtype,
             mode, static_cast<int32_t *>(const_cast<void *>(dot)),
             static_cast<int32_t *>(const_cast<void *>(don)), nullptr, nullptr, nullptr,
             stream_ptr, /*allow_tma=*/false, mir, mir + round256(t_bytes));
}

// ---------------------------------------------------------------------------
// One batch sharded over devices.  Sequences are independent, so shard g of G
// is the contiguous run [lo_g, hi_g) of sequences with lo_g = g (B / G) +
// min(g, B mod G): sizes differ by at most one, and the shards concatenate to
// the batch in order.  Each shard runs verify_host on its device, on a stream
// the library owns per (device, shard index); the outputs land in the
// caller's host arrays at the shard's offset.  Nothing crosses devices: no
// collective, no peer memory.
constexpr int kMaxShards = 64;

void shard_range(int64_t B, int32_t G, int32_t g, int64_t *lo, int64_t *hi) {
  const int64_t q = B / G, r = B % G;
  *lo = g * q + (g < r ? g : r);
  *hi = *lo + q + (g < r ? 1 : 0);
}

struct ShardStream {
  int dev;
  int shard;
  cudaStream_t stream;
};
std::vector<ShardStream> g_shard_streams;  // never destroyed while the process runs

// The library's stream for (dev, shard); dev must be current.
specv_status shard_stream(int dev, int shard, cudaStream_t *out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  for (const ShardStream &x : g_shard_streams)
    if (x.dev == dev && x.shard == shard) {
      *out = x.stream;
      return SPECV_OK;
    }
  cudaStream_t s = nullptr;
  const cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  g_shard_streams.push_back(ShardStream{dev, shard, s});
  *out = s;
  return SPECV_OK;
}

specv_status verify_sharded(const void *target, const void *draft, const int32_t *tokens,
                            const float *ua, const float *ur, const float *lam, int64_t B,
                            int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                            int32_t *out_tokens, int32_t *out_n, int32_t G,
                            const int32_t *devices) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n || !devices)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode) || G < 1 || G > kMaxShards) return SPECV_ERR_INVALID_ARG;
  int ndev = 0;
  cudaError_t e = cudaGetDeviceCount(&ndev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  for (int g = 0; g < G; ++g)
    if (devices[g] < 0 || devices[g] >= ndev) return SPECV_ERR_INVALID_ARG;
  int caller_dev = 0;
  if ((e = cudaGetDevice(&caller_dev)) != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  const size_t elem = dtype == SPECV_BF16 ? 2 : 4;
  const size_t row = (size_t)V * elem;
  specv_status status = SPECV_OK;
  cudaStream_t streams[kMaxShards] = {};
  // launch every shard (asynchronous: the devices work at the same time) ...
  for (int g = 0; g < G && status == SPECV_OK; ++g) {
    int64_t lo = 0, hi = 0;
    shard_range(B, G, g, &lo, &hi);
    if (hi == lo) continue;  // fewer sequences than shards
    if ((e = cudaSetDevice(devices[g])) != cudaSuccess) {
      note_cuda_error(e);
      (void)cudaGetLastError();
      status = SPECV_ERR_CUDA;
      break;
    }
    if ((status = shard_stream(devices[g], g, &streams[g])) != SPECV_OK) break;
    status = verify_host(static_cast<const char *>(target) + (size_t)lo * (K + 1) * row,
                         static_cast<const char *>(draft) + (size_t)lo * K * row, tokens + lo * K,
                         ua + lo * K, ur + lo, lam + lo, hi - lo, K, V, dtype, mode,
                         out_tokens + lo * (K + 1), out_n + lo, 0, streams[g]);
  }
  // ... then wait for all that were launched, so the outputs are in place on return
  for (int g = 0; g < G; ++g) {
    if (streams[g] == nullptr) continue;
    if ((e = cudaSetDevice(devices[g])) == cudaSuccess) e = cudaStreamSynchronize(streams[g]);
    if (e != cudaSuccess && status == SPECV_OK) {
      note_cuda_error(e);
      (void)cudaGetLastError();
      status = SPECV_ERR_CUDA;
    }
  }
  (void)cudaSetDevice(caller_dev);
  return status;
}

// ---------------------------------------------------------------------------
// Verify on host buffers, copying only the rows the verify step reaches.  The
// pages' loop stops at a sequence's first rejection, so the rows after it
// never influence the outputs; over a host link slower than HBM by a factor of
// about 30 those rows are most of the cost.  The batch goes over position by
// position: level i copies row pair (b, i) (at i = K the bonus row) of every
// sequence still alive, as one 2-D copy per run of live sequences, then the
// decision pass (specv_host_levels.cu) clears the flag of every sequence
// whose position i clearly rejects, and the host reads the flags back before
// the next level.  The sequences are dealt into kEeGroups interleaved groups
// (b mod kEeGroups), each with its own stream and level: while the host waits
// for one group's flags, the link carries another group's rows.  Rows never
// copied hold stale staging bytes; they all lie after their sequence's first
// rejection (the decision pass only stops a sequence on a rejection the verify
// step cannot see otherwise), so the ordinary verify step that follows on the
// staged batch never uses them.
constexpr int kEeGroups = 2;

specv_status verify_host_early_exit(const void *target, const void *draft, const int32_t *tokens,
                                    const float *ua, const float *ur, const float *lam, int64_t B,
                                    int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                    int32_t *out_tokens, int32_t *out_n, int64_t *out_h2d,
                                    int64_t *out_d2h, void *stream_ptr) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  const size_t elem = dtype == SPECV_BF16 ? 2 : 4;
  if ((uint64_t)B * (uint64_t)(2 * K + 1) > ((uint64_t)1 << 50) / elem / (uint64_t)V)
    return SPECV_ERR_NO_MEMORY;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status s = ensure_device(&sms, &l2);
  if (s != SPECV_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return SPECV_ERR_UNSUPPORTED;
  int dev = 0;
  (void)cudaGetDevice(&dev);

  // staging: the layout of verify_host, then the live flags (group-major:
  // group g's flags at g * Bg, Bg = ceil(B / kEeGroups))
  const int64_t Bg = (B + kEeGroups - 1) / kEeGroups;
  const size_t row = (size_t)V * elem;
  const size_t t_bytes = (size_t)B * (K + 1) * row, d_bytes = (size_t)B * K * row;
  const size_t bk4 = (size_t)B * K * 4, b4 = (size_t)B * 4, bk14 = (size_t)B * (K + 1) * 4;
  const size_t o_d = round256(t_bytes), o_tok = o_d + round256(d_bytes);
  const size_t o_ua = o_tok + round256(bk4), o_ur = o_ua + round256(bk4);
  const size_t o_lam = o_ur + round256(b4), o_ot = o_lam + round256(b4);
  const size_t o_on = o_ot + round256(bk14), o_al = o_on + round256(b4);
  const size_t flags = (size_t)(kEeGroups * Bg);
  const size_t need = o_al + round256(flags);
  HostPipe *hp = nullptr;
  if ((s = host_pipe(dev, stream, need, &hp)) != SPECV_OK) return s;
  if (hp->h_alive_bytes < flags) {
    if (hp->h_alive != nullptr) {  // no copy into it is pending, but drain the streams anyway
      (void)cudaStreamSynchronize(stream);
      (void)cudaStreamSynchronize(hp->copy);
      (void)cudaStreamSynchronize(hp->aux);
      (void)cudaFreeHost(hp->h_alive);
    }
    hp->h_alive = nullptr;
    hp->h_alive_bytes = 0;
    void *h = nullptr;
    if (cudaHostAlloc(&h, grow_to(flags), cudaHostAllocDefault) != cudaSuccess) {
      (void)cudaGetLastError();
      return SPECV_ERR_NO_MEMORY;
    }
    hp->h_alive = static_cast<unsigned char *>(h);
    hp->h_alive_bytes = grow_to(flags);
  }
  char *st = static_cast<char *>(hp->stage);
  unsigned char *alive = reinterpret_cast<unsigned char *>(st + o_al);
  unsigned char *h_alive = hp->h_alive;
  const char *tgt = static_cast<const char *>(target);
  const char *dft = static_cast<const char *>(draft);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  int64_t copied = (int64_t)(2 * bk4 + 2 * b4), read_back = (int64_t)(bk14 + b4);
  // Every host-to-device copy goes through one stream, in the order issued, so
  // that the link carries one group's rows while another group's decision pass
  // and read-back run (two copy streams would share the link and finish
  // together); group 0 decides on the caller's stream, group 1 on a second
  // stream of the pipe.  Events: ready[g] after group g's read-back, ready[2 + g]
  // after group g's copies.
  static_assert(kEeGroups >= 1 && kEeGroups <= 2, "one decision stream per group");
  cudaStream_t cs = hp->copy;
  cudaStream_t gs[2] = {stream, hp->aux};
  e = cudaMemcpyAsync(st + o_tok, tokens, bk4, h2d, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_ua, ua, bk4, h2d, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_ur, ur, b4, h2d, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st + o_lam, lam, b4, h2d, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(alive, 1, flags, stream);
  // the other streams start after these (and after earlier work on `stream`)
  if (e == cudaSuccess) e = cudaEventRecord(hp->start, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp->start, 0);
  for (int g = 1; g < kEeGroups && e == cudaSuccess; ++g) e = cudaStreamWaitEvent(gs[g], hp->start, 0);
  std::memset(h_alive, 1, flags);

  // the decision pass's geometry: one cluster per sequence
  const int vw = (int)(16 / elem);
  const int64_t G = (V + vw - 1) / vw;
  int S = specv::stream_cluster_size(Bg, (int64_t)row, G, sms);
  while (S > 1 && Bg * S > INT32_MAX) S /= 2;
  if (Bg * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
  const bool aligned = row % 16 == 0;
  int level[kEeGroups] = {};
  bool active[kEeGroups] = {};

  // level lv of group g: the live members' rows, then (below K) the decision
  // pass and the read-back of the group's flags, all on the group's stream
  auto issue = [&](int g) -> cudaError_t {
    const int64_t cnt = (B - g + kEeGroups - 1) / kEeGroups;  // members b = g + kEeGroups * j
    const unsigned char *hf = h_alive + g * Bg;
    const int lv = level[g];
    const size_t tp = (size_t)kEeGroups * (K + 1) * row, dp = (size_t)kEeGroups * K * row;
    int64_t live = 0;
    cudaError_t err = cudaSuccess;
    for (int64_t j0 = 0; j0 < cnt && err == cudaSuccess;) {
      if (!hf[j0]) {
        ++j0;
        continue;
      }
      int64_t j1 = j0 + 1;
      while (j1 < cnt && hf[j1]) ++j1;
      const size_t h = (size_t)(j1 - j0);
      const int64_t b0 = g + (int64_t)kEeGroups * j0;
      const size_t ot = ((size_t)b0 * (K + 1) + lv) * row;
      err = cudaMemcpy2DAsync(st + ot, tp, tgt + ot, tp, row, h, h2d, cs);
      copied += (int64_t)(h * row);
      if (err == cudaSuccess && lv < K) {
        const size_t od = ((size_t)b0 * K + lv) * row;
        err = cudaMemcpy2DAsync(st + o_d + od, dp, dft + od, dp, row, h, h2d, cs);
        copied += (int64_t)(h * row);
      }
      live += j1 - j0;
      j0 = j1;
    }
    if (err != cudaSuccess) return err;
    if (lv == K || live == 0) {
      active[g] = false;
      return cudaSuccess;
    }
    err = cudaEventRecord(hp->ready[2 + g], cs);  // the group's rows of this level are in
    if (err == cudaSuccess) err = cudaStreamWaitEvent(gs[g], hp->ready[2 + g], 0);
    if (err != cudaSuccess) return err;
    specv::LevelArgs la;
    la.target = st;
    la.draft = st + o_d;
    la.tokens = reinterpret_cast<const int32_t *>(st + o_tok);
    la.u_accept = reinterpret_cast<const float *>(st + o_ua);
    la.lam = reinterpret_cast<const float *>(st + o_lam);
    la.alive = alive + g * Bg;
    la.count = cnt;
    la.group = g;
    la.n_groups = kEeGroups;
    la.K = K;
    la.V = V;
    la.level = lv;
    la.num_groups = (int)G;
    la.groups_per_slice = (int)((G + S - 1) / S);
    err = specv::level_launch(la, dtype == SPECV_BF16, mode, aligned, S, gs[g]);
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(h_alive + g * Bg, alive + g * Bg, (size_t)cnt, cudaMemcpyDeviceToHost,
                            gs[g]);
    if (err == cudaSuccess) err = cudaEventRecord(hp->ready[g], gs[g]);
    read_back += cnt;
    return err;
  };
  for (int g = 0; g < kEeGroups; ++g) {
    level[g] = 0;
    active[g] = g < B;
  }
  for (int g = 0; g < kEeGroups && e == cudaSuccess; ++g)
    if (active[g]) e = issue(g);
  for (bool any = true; any && e == cudaSuccess;) {
    any = false;
    for (int g = 0; g < kEeGroups && e == cudaSuccess; ++g) {
      if (!active[g]) continue;
      any = true;
      e = cudaEventSynchronize(hp->ready[g]);  // the group's flags are on the host
      if (e == cudaSuccess) {
        ++level[g];
        e = issue(g);
      }
    }
  }
  // the verify step on the staged batch once every copy is in
  if (e == cudaSuccess) e = cudaEventRecord(hp->ready[4], cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, hp->ready[4], 0);
  for (int g = 1; g < kEeGroups && e == cudaSuccess; ++g) {
    e = cudaEventRecord(hp->ready[g], gs[g]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, hp->ready[g], 0);
  }
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  s = run(st, st + o_d, reinterpret_cast<const int32_t *>(st + o_tok),
          reinterpret_cast<const float *>(st + o_ua), reinterpret_cast<const float *>(st + o_ur),
          reinterpret_cast<const float *>(st + o_lam), B, K, V, dtype, mode,
          reinterpret_cast<int32_t *>(st + o_ot), reinterpret_cast<int32_t *>(st + o_on), nullptr,
          nullptr, nullptr, stream);
  if (s != SPECV_OK) return s;
  e = cudaMemcpyAsync(out_tokens, st + o_ot, bk14, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_n, st + o_on, b4, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (out_h2d) *out_h2d = copied;
  if (out_d2h) *out_d2h = read_back;
  return SPECV_OK;
}

// An NVTX range named after the entry point around its host work and launches:
// visible on the timeline of NVIDIA's profilers, a no-op when none is attached.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace

extern "C" {

specv_status specv_verify(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *lambda, int64_t B, int32_t K,
                          int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                          int32_t *out_n_accepted, void *stream) {
  NvtxRange range("specv_verify");
  return run(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda, B, K, V,
             dtype, mode, out_tokens, out_n_accepted, nullptr, nullptr, nullptr, stream);
}

specv_status specv_verify_host(const void *target_logits, const void *draft_logits,
                               const int32_t *draft_tokens, const float *u_accept,
                               const float *u_resample, const float *lambda, int64_t B, int32_t K,
                               int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                               int32_t *out_n_accepted, int32_t chunks, void *stream) {
  NvtxRange range("specv_verify_host");
  return verify_host(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda, B,
                     K, V, dtype, mode, out_tokens, out_n_accepted, chunks, stream);
}

specv_status specv_verify_host_direct(const void *target_logits, const void *draft_logits,
                                      const int32_t *draft_tokens, const float *u_accept,
                                      const float *u_resample, const float *lambda, int64_t B,
                                      int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                      int32_t *out_tokens, int32_t *out_n_accepted,
                                      void *stream) {
  NvtxRange range("specv_verify_host_direct");
  return verify_host_direct(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                            lambda, B, K, V, dtype, mode, out_tokens, out_n_accepted, stream);
}

specv_status specv_verify_host_early_exit(const void *target_logits, const void *draft_logits,
                                          const int32_t *draft_tokens, const float *u_accept,
                                          const float *u_resample, const float *lambda,
                                          int64_t B, int32_t K, int32_t V, specv_dtype dtype,
                                          specv_mode mode, int32_t *out_tokens,
                                          int32_t *out_n_accepted, int64_t *out_h2d_bytes,
                                          int64_t *out_d2h_bytes, void *stream) {
  NvtxRange range("specv_verify_host_early_exit");
  return verify_host_early_exit(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                                lambda, B, K, V, dtype, mode, out_tokens, out_n_accepted,
                                out_h2d_bytes, out_d2h_bytes, stream);
}

specv_status specv_shard_bounds(int64_t B, int32_t n_shards, int32_t shard, int64_t *lo,
                                int64_t *hi) {
  if (!lo || !hi || B < 0 || n_shards < 1 || n_shards > kMaxShards || shard < 0 ||
      shard >= n_shards)
    return SPECV_ERR_INVALID_ARG;
  shard_range(B, n_shards, shard, lo, hi);
  return SPECV_OK;
}

specv_status specv_verify_sharded_host(const void *target_logits, const void *draft_logits,
                                       const int32_t *draft_tokens, const float *u_accept,
                                       const float *u_resample, const float *lambda, int64_t B,
                                       int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                       int32_t *out_tokens, int32_t *out_n_accepted,
                                       int32_t n_shards, const int32_t *devices) {
  NvtxRange range("specv_verify_sharded_host");
  return verify_sharded(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda,
                        B, K, V, dtype, mode, out_tokens, out_n_accepted, n_shards, devices);
}

specv_status specv_verify_debug(const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *u_accept,
                                const float *u_resample, const float *lambda, int64_t B,
                                int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                int32_t *out_tokens, int32_t *out_n_accepted,
                                float *out_ptilde_at_x, float *out_q_at_x, float *out_lse,
                                void *stream) {
  if (mode == SPECV_GREEDY) return SPECV_ERR_UNSUPPORTED;  // no probabilities to report
  NvtxRange range("specv_verify_debug");
  return run(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda, B, K, V,
             dtype, mode, out_tokens, out_n_accepted, out_ptilde_at_x, out_q_at_x, out_lse,
             stream);
}

specv_status specv_plan(int64_t B, int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                        int32_t *kernel, int32_t *cluster, int64_t *ctas,
                        int64_t *workspace_bytes) {
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess && v > 0) l2 = v;
    (void)cudaGetLastError();
  } else {
    (void)cudaGetLastError();
  }
  Plan p;
  specv_status s = make_plan(B, K, V, dtype, mode, sms, l2, true, &p);
  if (s != SPECV_OK) return s;
  if (kernel) *kernel = p.kernel;
  if (cluster) *cluster = p.cluster;
  if (ctas) *ctas = p.ctas;
  if (workspace_bytes) *workspace_bytes = p.ws_bytes;
  return SPECV_OK;
}

specv_status specv_plan_flags(int64_t B, int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                              uint32_t *flags) {
  if (!flags || !sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
    (void)cudaGetLastError();
  } else {
    (void)cudaGetLastError();
  }
  Plan p;
  specv_status s = make_plan(B, K, V, dtype, mode, sms, l2, true, &p);
  if (s != SPECV_OK) return s;
  *flags = (p.early_exit ? SPECV_PLAN_EARLY_EXIT : 0u) | (p.split ? SPECV_PLAN_SPLIT_DRAWS : 0u);
  return SPECV_OK;
}

specv_status specv_verify_tree(const void *target_logits, const void *draft_logits,
                               const int32_t *parent, const int32_t *draft_row,
                               const int32_t *tokens, const float *u_accept,
                               const float *u_resample, const float *lambda, int64_t B, int32_t N,
                               int32_t M, int32_t V, specv_dtype dtype, specv_mode mode,
                               int32_t *out_tokens, int32_t *out_path, int32_t *out_n,
                               void *stream) {
  NvtxRange range("specv_verify_tree");
  if (!target_logits || !parent || !draft_row || !tokens || !u_accept || !u_resample || !lambda ||
      !out_tokens || !out_path || !out_n || (M > 0 && !draft_logits))
    return SPECV_ERR_INVALID_ARG;
  if (B < 1 || N < 0 || N > kMaxK || M < 0 || V < 1) return SPECV_ERR_INVALID_ARG;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (mode != SPECV_PROB_MIX && mode != SPECV_LOGIT_MIX) return SPECV_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 62;
  if (B > lim / (N + 1) || B * (N + 1) > lim / V || (M > 0 && B * (int64_t)M > lim / V))
    return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status st = ensure_device(&sms, &l2);
  if (st != SPECV_OK) return st;
  const int bf16 = dtype == SPECV_BF16;
  const int elem = bf16 ? 2 : 4;
  const int vw = 16 / elem;
  const int64_t row_bytes = (int64_t)V * elem;
  const int64_t G = (V + vw - 1) / vw;
  const int64_t P = B * (N + 1);
  const bool aligned = ((uintptr_t)target_logits % 16 == 0) &&
                       (M == 0 || (uintptr_t)draft_logits % 16 == 0) && (row_bytes % 16 == 0);
  // cluster size: the streaming row kernel's rule
  int S = cluster_from_env();
  if (S == 0) {
    S = specv::stream_cluster_size(P, row_bytes, G, sms);
  }
  while (S > 1 && P * S > INT32_MAX) S /= 2;
  if (P * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  (void)cudaGetDevice(&dev);
  const size_t data_bytes = (size_t)round16(P * 16);
  unsigned *cnt = nullptr;
  void *wdata = nullptr;
  void *ws = nullptr;
  cudaError_t e = cudaSuccess;
  const bool per_call = !cached_workspace(dev, s, B, data_bytes, &cnt, &wdata);
  if (per_call) {
    e = cudaMallocAsync(&ws, data_bytes + (size_t)round16(B * 4), s);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      (void)cudaGetLastError();
      return SPECV_ERR_NO_MEMORY;
    }
    cnt = static_cast<unsigned *>(ws);
    wdata = static_cast<char *>(ws) + round16(B * 4);
    e = cudaMemsetAsync(cnt, 0, (size_t)B * sizeof(unsigned), s);
  }
  specv::TreeArgs a;
  a.target = target_logits;
  a.draft = draft_logits ? draft_logits : target_logits;  // M == 0: never read
  a.parent = parent;
  a.draft_row = draft_row;
  a.tokens = tokens;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.lam = lambda;
  a.B = B;
  a.N = N;
  a.M = M;
  a.V = V;
  a.out_tokens = out_tokens;
  a.out_path = out_path;
  a.out_n = out_n;
  a.ws_stats = static_cast<float4 *>(wdata);
  a.ws_count = cnt;
  a.num_groups = (int)G;
  a.groups_per_slice = (int)((G + S - 1) / S);
  specv::rows_segments(a.groups_per_slice, &a.seg_tiles, &a.segs_per_slice);
  if (e == cudaSuccess) e = specv::tree_launch(a, bf16, mode, aligned, S, P * S, s);
  if (per_call) {
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

specv_status specv_acceptance_rates(const void *target_logits, const void *draft_logits,
                                    const float *lambda, int64_t B, int32_t K, int32_t V,
                                    specv_dtype dtype, specv_mode mode, float *out_alpha,
                                    void *stream) {
  NvtxRange range("specv_acceptance_rates");
  if (!target_logits || !draft_logits || !lambda || !out_alpha) return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  if (mode == SPECV_GREEDY) return SPECV_ERR_UNSUPPORTED;  // greedy has no p~ to overlap with q
  int sms = kDefaultSMs;
  int64_t l2 = kDefaultL2;
  specv_status s = ensure_device(&sms, &l2);
  if (s != SPECV_OK) return s;
  const int bf16 = dtype == SPECV_BF16;
  const int elem = bf16 ? 2 : 4;
  const int vw = 16 / elem;
  const int64_t row_bytes = (int64_t)V * elem;
  const int64_t G = (V + vw - 1) / vw;
  const int64_t Q = B * K;  // drafted positions
  const bool aligned = ((uintptr_t)target_logits % 16 == 0) && ((uintptr_t)draft_logits % 16 == 0) &&
                       (row_bytes % 16 == 0);
  // Cluster size: the smallest power of two (<= 16) that keeps one CTA's
  // slice of the pair within 128 KiB (so the second pass finds it in L2) and
  // gives >= 8 CTAs per SM, without going under 4 KiB of a row per CTA.
  int S = cluster_from_env();
  if (S == 0) {
    S = 1;
    while (S < specv::kMaxCluster && row_bytes / (2 * S) >= 4096 &&
           (Q * S < 8LL * sms || 2 * row_bytes / S > 128 * 1024))
      S *= 2;
  }
  while (S > 1 && Q * S > INT32_MAX) S /= 2;
  if (Q * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
  specv::AlphaArgs a;
  a.target = target_logits;
  a.draft = draft_logits;
  a.lam = lambda;
  a.B = B;
  a.K = K;
  a.V = V;
  a.out_alpha = out_alpha;
  a.num_groups = (int)G;
  a.groups_per_slice = (int)((G + S - 1) / S);
  const cudaError_t e = specv::alpha_launch(a, bf16, mode, aligned, S, Q * S,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

int32_t specv_choose_k(double alpha, double cost_draft, double cost_verify_fixed,
                       double cost_verify_per_token, int32_t k_min, int32_t k_max) {
  if (!(alpha >= 0.0 && alpha <= 1.0)) return -1;
  if (k_min < 1 || k_max < k_min || k_max > kMaxK) return -1;
  if (!(cost_draft >= 0.0) || !(cost_verify_fixed >= 0.0) || !(cost_verify_per_token >= 0.0))
    return -1;
  int32_t best_k = k_min;
  double best = -1.0;
  for (int32_t k = k_min; k <= k_max; ++k) {
    // expected tokens of one step: 1 + a + ... + a^k (the accepted prefix and
    // the token drawn at its end), over the step's cost
    double tokens = 0.0, ak = 1.0;
    for (int32_t j = 0; j <= k; ++j) {
      tokens += ak;
      ak *= alpha;
    }
    const double cost = cost_verify_fixed + (double)k * (cost_draft + cost_verify_per_token);
    if (!(cost > 0.0)) return -1;
    const double rate = tokens / cost;
    if (rate > best) {
      best = rate;
      best_k = k;
    }
  }
  return best_k;
}

specv_status specv_release_stream(void *stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return SPECV_ERR_UNSUPPORTED;
  std::vector<void *> dev_bufs, host_bufs;
  std::vector<cudaStream_t> copy_streams;
  std::vector<cudaEvent_t> events;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (size_t k = 0; k < g_ws.size();) {
      Workspace &w = g_ws[k];
      if (w.dev == dev && w.stream == s) {
        if (w.count) dev_bufs.push_back(w.count);
        if (w.data) dev_bufs.push_back(w.data);
        for (void *p : w.superseded) dev_bufs.push_back(p);
        g_ws.erase(g_ws.begin() + (std::ptrdiff_t)k);
      } else {
        ++k;
      }
    }
    for (size_t k = 0; k < g_pipes.size();) {
      HostPipe *hp = g_pipes[k];
      if (hp->dev == dev && hp->stream == s) {
        if (hp->stage) dev_bufs.push_back(hp->stage);
        if (hp->h_alive) host_bufs.push_back(hp->h_alive);
        copy_streams.push_back(hp->copy);
        copy_streams.push_back(hp->aux);
        events.push_back(hp->start);
        for (int c = 0; c < kHostMaxChunks; ++c) events.push_back(hp->ready[c]);
        delete hp;
        g_pipes.erase(g_pipes.begin() + (std::ptrdiff_t)k);
      } else {
        ++k;
      }
    }
  }
  // the stream's queued work may still use the buffers: let it finish first
  e = cudaStreamSynchronize(s);
  for (cudaStream_t c : copy_streams)
    if (e == cudaSuccess) e = cudaStreamSynchronize(c);
  for (void *p : dev_bufs) (void)cudaFree(p);
  for (void *p : host_bufs) (void)cudaFreeHost(p);
  for (cudaEvent_t ev : events) (void)cudaEventDestroy(ev);
  for (cudaStream_t c : copy_streams) (void)cudaStreamDestroy(c);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

const char *specv_status_string(specv_status status) {
  switch (status) {
    case SPECV_OK: return "SPECV_OK";
    case SPECV_ERR_INVALID_ARG: return "SPECV_ERR_INVALID_ARG";
    case SPECV_ERR_UNSUPPORTED: return "SPECV_ERR_UNSUPPORTED";
    case SPECV_ERR_CUDA: return "SPECV_ERR_CUDA";
    case SPECV_ERR_NO_MEMORY: return "SPECV_ERR_NO_MEMORY";
  }
  return "SPECV_ERR_UNKNOWN";
}

const char *specv_last_cuda_error(void) { return g_last_cuda_error; }

int32_t specv_version(void) { return 100; }

}  // extern "C"
