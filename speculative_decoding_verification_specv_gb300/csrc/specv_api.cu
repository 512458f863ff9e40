// specv_api.cu -- the C ABI of libspecv.so (declared in include/specv.h).
//
// Host-side work only: argument validation, the launch plan (which kernel,
// cluster size, grid), the per-call scratch workspace and the launches.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "specv.h"
#include "specv_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultSMs = 152;        // used by specv_plan when no device is visible
constexpr int kTileSmemBudget = 48 * 1024;
constexpr int kTileMaxV = 256;
constexpr int kTileMinSeqs = 4;
constexpr int kTileMaxSeqs = 64;
constexpr int32_t kMaxK = 4096;

struct DeviceState {
  bool ready = false;
  cudaError_t err = cudaSuccess;
  int sms = kDefaultSMs;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
thread_local char g_last_cuda_error[256] = "";

void note_cuda_error(cudaError_t e) {
  std::strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
  g_last_cuda_error[sizeof(g_last_cuda_error) - 1] = '\0';
}

// One-time per-device set-up: opt the kernels into 16-CTA clusters and the
// tile kernel into its shared-memory size; read the SM count.
specv_status ensure_device(int *sms_out) {
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
    int major = 0, cluster_ok = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    if (major < 10 || !cluster_ok) return SPECV_ERR_UNSUPPORTED;
    if ((e = specv::rows_prepare()) != cudaSuccess || (e = specv::tile_prepare(kTileSmemBudget)) != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    st.sms = sms;
    st.ready = true;
  }
  if (sms_out) *sms_out = st.sms;
  return SPECV_OK;
}

struct Plan {
  int kernel;            // 0 tile, 1 rows
  int cluster;           // CTAs per cluster (rows kernel)
  int64_t ctas;          // CTAs of the rows kernel (tile kernel: tiles)
  int64_t ws_bytes;      // scratch bytes
  int tile_seqs;
  int smem_t, smem_d, smem_total;
  int groups_per_slice, num_groups;
};

int64_t round16(int64_t x) { return (x + 15) / 16 * 16; }

bool sizes_ok(int64_t B, int32_t K, int32_t V, int dtype, int mode) {
  if (B < 1 || K < 1 || K > kMaxK || V < 1) return false;
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return false;
  if (mode != SPECV_PROB_MIX && mode != SPECV_LOGIT_MIX) return false;
  const int64_t lim = (int64_t)1 << 62;
  if (B > lim / (K + 1) || B * (K + 1) > lim / V) return false;
  return true;
}

int cluster_from_env() {
  const char *s = std::getenv("SPECV_CLUSTER_SIZE");
  if (!s || !*s) return 0;
  int v = std::atoi(s);
  return (v == 1 || v == 2 || v == 4 || v == 8 || v == 16) ? v : 0;
}

// The launch plan.  Short rows whose whole sequences fit a shared-memory tile
// go to the tile kernel; everything else to the cluster row kernel, with the
// cluster size doubled (up to 16) while the grid has fewer than 4 CTAs per SM
// and each CTA would still stream at least 4 KiB of every row.
specv_status make_plan(int64_t B, int32_t K, int32_t V, int dtype, int sms, Plan *p) {
  const int elem = dtype == SPECV_BF16 ? 2 : 4;
  std::memset(p, 0, sizeof(*p));
  const int64_t seq_bytes = (int64_t)(2 * K + 1) * V * elem + (int64_t)(K + 1) * 16;
  if (V <= kTileMaxV && seq_bytes * kTileMinSeqs + 64 <= kTileSmemBudget) {
    int ts = (int)((kTileSmemBudget - 64) / seq_bytes);
    if (ts > kTileMaxSeqs) ts = kTileMaxSeqs;
    if (ts > B) ts = (int)B;
    p->kernel = 0;
    p->cluster = 1;
    p->tile_seqs = ts;
    p->smem_t = (int)round16((int64_t)ts * (K + 1) * V * elem);
    p->smem_d = (int)round16((int64_t)ts * K * V * elem);
    p->smem_total = p->smem_t + p->smem_d + ts * (K + 1) * 16;
    p->ctas = (B + ts - 1) / ts;  // tiles
    p->ws_bytes = 0;
    return SPECV_OK;
  }
  const int64_t P = B * (K + 1);
  const int vw = 16 / elem;
  const int64_t row_bytes = (int64_t)V * elem;
  int S = cluster_from_env();
  if (S == 0) {
    S = 1;
    while (S < specv::kMaxCluster && P * S < 4LL * sms && row_bytes / (2 * S) >= 4096) S *= 2;
  }
  while (S > 1 && P * S > INT32_MAX) S /= 2;
  if (P * S > INT32_MAX) return SPECV_ERR_UNSUPPORTED;
  p->kernel = 1;
  p->cluster = S;
  p->ctas = P * S;
  p->num_groups = (int)((V + vw - 1) / vw);
  p->groups_per_slice = (p->num_groups + S - 1) / S;
  p->ws_bytes = round16(P * 16) + round16(B * 4);
  return SPECV_OK;
}

specv_status run(const void *target, const void *draft, const int32_t *tokens, const float *ua,
                 const float *ur, const float *lam, int64_t B, int32_t K, int32_t V,
                 specv_dtype dtype, specv_mode mode, int32_t *out_tokens, int32_t *out_n,
                 float *dbg_ptilde, float *dbg_q, float *dbg_lse, void *stream_ptr) {
  if (!target || !draft || !tokens || !ua || !ur || !lam || !out_tokens || !out_n)
    return SPECV_ERR_INVALID_ARG;
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  specv_status s = ensure_device(&sms);
  if (s != SPECV_OK) return s;
  Plan p;
  if ((s = make_plan(B, K, V, dtype, sms, &p)) != SPECV_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int bf16 = dtype == SPECV_BF16;
  const int elem = bf16 ? 2 : 4;
  cudaError_t e;
  if (p.kernel == 0) {
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
    const int per_sm = specv::tile_blocks_per_sm(bf16, mode, p.smem_total);
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > p.ctas) grid = p.ctas;
    e = specv::tile_launch(a, bf16, mode, grid, p.smem_total, stream);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      return SPECV_ERR_CUDA;
    }
    return SPECV_OK;
  }
  void *ws = nullptr;
  e = cudaMallocAsync(&ws, (size_t)p.ws_bytes, stream);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    (void)cudaGetLastError();
    return SPECV_ERR_NO_MEMORY;
  }
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
  a.ws_stats = static_cast<float4 *>(ws);
  a.ws_count = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + round16(B * (K + 1) * 16));
  a.dbg_ptilde = dbg_ptilde;
  a.dbg_q = dbg_q;
  a.dbg_lse = dbg_lse;
  a.groups_per_slice = p.groups_per_slice;
  a.num_groups = p.num_groups;
  const bool aligned = ((uintptr_t)target % 16 == 0) && ((uintptr_t)draft % 16 == 0) &&
                       ((int64_t)V * elem % 16 == 0);
  e = cudaMemsetAsync(a.ws_count, 0, (size_t)B * sizeof(unsigned), stream);
  if (e == cudaSuccess) e = specv::rows_launch(a, bf16, mode, aligned, p.cluster, p.ctas, stream);
  const cudaError_t ef = cudaFreeAsync(ws, stream);
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

}  // namespace

extern "C" {

specv_status specv_verify(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *lambda, int64_t B, int32_t K,
                          int32_t V, specv_dtype dtype, specv_mode mode, int32_t *out_tokens,
                          int32_t *out_n_accepted, void *stream) {
  return run(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda, B, K, V,
             dtype, mode, out_tokens, out_n_accepted, nullptr, nullptr, nullptr, stream);
}

specv_status specv_verify_debug(const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *u_accept,
                                const float *u_resample, const float *lambda, int64_t B,
                                int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                                int32_t *out_tokens, int32_t *out_n_accepted,
                                float *out_ptilde_at_x, float *out_q_at_x, float *out_lse,
                                void *stream) {
  return run(target_logits, draft_logits, draft_tokens, u_accept, u_resample, lambda, B, K, V,
             dtype, mode, out_tokens, out_n_accepted, out_ptilde_at_x, out_q_at_x, out_lse,
             stream);
}

specv_status specv_plan(int64_t B, int32_t K, int32_t V, specv_dtype dtype, specv_mode mode,
                        int32_t *kernel, int32_t *cluster, int64_t *ctas,
                        int64_t *workspace_bytes) {
  if (!sizes_ok(B, K, V, dtype, mode)) return SPECV_ERR_INVALID_ARG;
  int sms = kDefaultSMs;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      sms = v;
  } else {
    (void)cudaGetLastError();
  }
  Plan p;
  specv_status s = make_plan(B, K, V, dtype, sms, &p);
  if (s != SPECV_OK) return s;
  if (kernel) *kernel = p.kernel;
  if (cluster) *cluster = p.cluster;
  if (ctas) *ctas = p.kernel == 0 ? p.ctas : p.ctas;
  if (workspace_bytes) *workspace_bytes = p.ws_bytes;
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
