// specv_internal.h -- launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

// Records the CUDA error behind a SPECV_ERR_CUDA for specv_last_cuda_error
// (per host thread).
void note_cuda_error(cudaError_t e);

constexpr int kRowThreads = 256;   // threads per CTA of the cluster row kernel
constexpr int kMaxCluster = 16;    // largest cluster (non-portable size, opt-in)
constexpr int kTileThreads = 256;  // threads per CTA of the small-vocabulary kernel
constexpr int kTmaTileThreads = 256;  // threads per CTA of the TMA tile kernel
constexpr int kTmaTileLanes = 4;      // stage-B lanes per sequence of the TMA tile kernel
constexpr int kTmaTileMaxSeqs = kTmaTileThreads / kTmaTileLanes;  // sequences per TMA tile
constexpr int kResidentChunkGroups = 1024;  // 16-byte groups per TMA chunk (16 KiB per row)
constexpr int kResidentMaxChunks = 8;       // chunks per row slice (128 KiB per row at most)

// Sampler segments of the streaming row kernel.  A CTA's slice of a row is cut
// into segments of seg_tiles * kSegGroups consecutive 16-byte groups (the last
// one may be short), at most kMaxSegs per slice; a warp reads a tile of
// kSegGroups groups as kSegLaneGroups coalesced 16-byte loads per lane.
constexpr int kSegLaneGroups = 4;
constexpr int kSegGroups = 32 * kSegLaneGroups;
constexpr int kMaxSegs = 512;

// Segment geometry of a slice of `groups` groups read in tiles of tile_groups:
// the fewest whole tiles per segment that keep the count within kMaxSegs.
inline void segment_geometry(int64_t groups, int tile_groups, int *seg_tiles, int *nseg) {
  const int64_t tiles = (groups + tile_groups - 1) / tile_groups;
  const int64_t per_seg = (tiles + kMaxSegs - 1) / kMaxSegs;
  *seg_tiles = (int)(per_seg < 1 ? 1 : per_seg);
  const int64_t seg_groups = (int64_t)*seg_tiles * tile_groups;
  *nseg = (int)((groups + seg_groups - 1) / seg_groups);
}
inline void rows_segments(int groups_per_slice, int *seg_tiles, int *segs_per_slice) {
  segment_geometry(groups_per_slice, kSegGroups, seg_tiles, segs_per_slice);
}

// Cluster size of the streaming row kernels (verify, greedy, tree) for P
// positions of rows of row_bytes bytes (groups 16-byte groups) on `sms` SMs.
// The smallest power of two (<= kMaxCluster) that gives the grid >= 4 CTAs per
// SM and each CTA <= 512 KiB of (target + draft) slice, without going under
// 4 KiB of a row per CTA.  When that grid is at most two waves of 4 CTAs per
// SM, the size (any 1..kMaxCluster within the same slice limits) that
// minimises waves x (slice length + a fixed cost per CTA of kCtaFixedGroups
// groups) instead: a badly quantised wave costs a whole extra slice time (at
// 192 positions S = 3 fills one wave where S = 4 needs two).
constexpr int64_t kCtaFixedGroups = 2048;
inline int stream_cluster_size(int64_t P, int64_t row_bytes, int64_t groups, int sms) {
  int S = 1;
  while (S < kMaxCluster && row_bytes / (2 * S) >= 4096 &&
         (P * S < 4LL * sms || 2 * row_bytes / S > 512 * 1024))
    S *= 2;
  const int64_t slots = 4LL * sms;
  if (P * S > 2 * slots) return S;
  auto cost = [&](int s) {
    return ((P * s + slots - 1) / slots) * ((groups + s - 1) / s + kCtaFixedGroups);
  };
  int best = S;
  for (int s = 1; s <= kMaxCluster; ++s) {
    if (s > 1 && row_bytes / (2 * s) < 4096) continue;
    if (2 * row_bytes / s > 512 * 1024) continue;
    if (cost(s) < cost(best)) best = s;
  }
  return best;
}

// Arguments of the cluster row kernel (one cluster per (sequence, position)).
struct RowArgs {
  const void *target;        // [B][K+1][V]
  const void *draft;         // [B][K][V]
  const int32_t *tokens;     // [B][K]
  const float *u_accept;     // [B][K]
  const float *u_resample;   // [B]
  const float *lam;          // [B]
  int64_t B;
  int K;
  int V;
  int32_t *out_tokens;       // [B][K+1]
  int32_t *out_n;            // [B]
  float4 *ws_stats;          // scratch [B][K+1]: (mA, sA, mB, sB) per position
  unsigned *ws_count;        // scratch [B]: positions published so far (zeroed per call)
  float *dbg_ptilde;         // optional [B][K]
  float *dbg_q;              // optional [B][K]
  float *dbg_lse;            // optional [B][K+1][2]
  int groups_per_slice;      // 16-byte groups of a row handled by one CTA
  int num_groups;            // ceil(V / elements per 16 bytes)
  int seg_tiles;             // sampler segment = seg_tiles * kSegGroups groups
  int segs_per_slice;        // segments of one CTA's slice (<= kMaxSegs)
  float2 *ws_seg;            // optional scratch [B][S][segs_per_slice]: (max, sum-exp) of the
                             // bonus row's segments, written in phase 1 (null: the sampler
                             // reads the bonus row again)
  int defer_sampling;        // 1: the last cluster stops after the decisions; rows_sample
                             // draws the tokens in a second launch
  unsigned *ws_reject = nullptr;  // optional scratch [B] (zero at entry, left zero): early exit.
                                  // K + 1 - j for the earliest position j whose own acceptance
                                  // test is known to reject; positions after it skip their rows
  void *mirror_target = nullptr;  // optional device copies [B][K+1][V] / [B][K][V] (aligned
  void *mirror_draft = nullptr;   // rows): the stream stores what it reads there, and the
                                  // token draws read the rows back from them
  int pos_major = 0;         // 1: the grid runs position-major (all sequences' position 0, then
                             // position 1, ...), so that later positions of a sequence start
                             // after its earlier ones have published their decisions
  // rows_sample only: the statistics launch's geometry (for the bonus segments)
  int stats_cluster;
  int stats_groups_per_slice;
  int stats_seg_tiles;
  int stats_segs_per_slice;
};

// Arguments of the small-vocabulary tile kernel (a CTA holds whole sequences).
struct TileArgs {
  const void *target;
  const void *draft;
  const int32_t *tokens;
  const float *u_accept;
  const float *u_resample;
  const float *lam;
  int64_t B;
  int K;
  int V;
  int32_t *out_tokens;
  int32_t *out_n;
  float *dbg_ptilde;
  float *dbg_q;
  float *dbg_lse;
  int tile_seqs;             // sequences per tile
  int64_t num_tiles;
  int vec_copy;              // 1: tiles start on 16-byte boundaries and span whole vectors
  int smem_target_bytes;     // bytes of a staged target block (16-byte padded)
  int smem_draft_bytes;      // bytes of a staged draft block (16-byte padded)
};

// Arguments of the resident cluster row kernel (slices staged in shared memory,
// sampling decided per position).
struct ResArgs {
  const void *target;        // [B][K+1][V]
  const void *draft;         // [B][K][V]
  const int32_t *tokens;     // [B][K]
  const float *u_accept;     // [B][K]
  const float *u_resample;   // [B]
  const float *lam;          // [B]
  int64_t B;
  int K;
  int V;
  int32_t *out_tokens;       // [B][K+1]
  int32_t *out_n;            // [B]
  int2 *rec;                 // scratch [B][K+1]: (status, token) per position
  unsigned *count;           // scratch [B]: positions published so far (zeroed per call)
  float *dbg_ptilde;         // optional [B][K]
  float *dbg_q;              // optional [B][K]
  float *dbg_lse;            // optional [B][K+1][2]
  int groups_per_slice;      // 16-byte groups of a row staged by one CTA
  int num_groups;            // V / elements per 16 bytes (V * sizeof(dtype) % 16 == 0)
};

cudaError_t resident_prepare(int max_smem);
cudaError_t resident_launch(const ResArgs &a, int dtype_bf16, int mode, int S, int64_t grid,
                            int smem, cudaStream_t stream);

// Arguments of the acceptance-probability kernel (one cluster per drafted
// position b*K + i).
struct AlphaArgs {
  const void *target;        // [B][K+1][V]
  const void *draft;         // [B][K][V]
  const float *lam;          // [B]
  int64_t B;
  int K;
  int V;
  float *out_alpha;          // [B][K]
  int groups_per_slice;      // 16-byte groups of a row handled by one CTA
  int num_groups;            // ceil(V / elements per 16 bytes)
};
cudaError_t alpha_prepare();
cudaError_t alpha_launch(const AlphaArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                         int64_t grid, cudaStream_t stream);

// Arguments of the tree-verification kernel (one cluster per tree node b*(N+1) + u).
struct TreeArgs {
  const void *target;        // [B][N+1][V]: target row of every node
  const void *draft;         // [B][M][V]: draft rows
  const int32_t *parent;     // [B][N+1]: parent node (-1 at the root)
  const int32_t *draft_row;  // [B][N+1]: draft row a node's children were drawn from, or -1
  const int32_t *tokens;     // [B][N+1]: token of every node (entry 0 unused)
  const float *u_accept;     // [B][N+1]: uniform of every node's test (entry 0 unused)
  const float *u_resample;   // [B]
  const float *lam;          // [B]
  int64_t B;
  int N;
  int M;
  int V;
  int32_t *out_tokens;       // [B][N+1]
  int32_t *out_path;         // [B][N+1]
  int32_t *out_n;            // [B]
  float4 *ws_stats;          // scratch [B][N+1]: (mA, sA, mB, sB) of every node
  unsigned *ws_count;        // scratch [B]: nodes published so far (zero at entry, left zero)
  int groups_per_slice;
  int num_groups;
  int seg_tiles;
  int segs_per_slice;
};
cudaError_t tree_prepare();
cudaError_t tree_launch(const TreeArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                        int64_t grid, cudaStream_t stream);

cudaError_t rows_prepare();
cudaError_t rows_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                        int64_t grid, cudaStream_t stream);
// The sequence-cluster kernel: one cluster of S CTAs per sequence (grid B * S)
// streams every position of its sequence, decides it and draws its token in
// one launch (grids of about one wave); K + 1 <= kSeqMaxPositions, device
// memory only (aligned rows are staged with asynchronous copies).
constexpr int kSeqMaxPositions = 64;
cudaError_t rows_seq_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                            cudaStream_t stream);
// The deferred token draws: one cluster of S CTAs per sequence (grid B * S),
// after a rows_launch with defer_sampling = 1 on the same stream.
cudaError_t rows_sample_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                               int64_t grid, cudaStream_t stream);

// Arguments of the host-buffer call's decision pass (one cluster per
// sequence of one group): the group holds sequences b = group + n_groups * j,
// j in [0, count); position `level` of every one with alive[j] != 0 is
// decided, and alive[j] is cleared when it clearly rejects.
struct LevelArgs {
  const void *target;        // [B][K+1][V] (staged; rows up to `level` present for live sequences)
  const void *draft;         // [B][K][V]
  const int32_t *tokens;     // [B][K]
  const float *u_accept;     // [B][K]
  const float *lam;          // [B]
  unsigned char *alive;      // [count]: the group's flags
  int64_t count;             // sequences in the group
  int group;
  int n_groups;
  int K;
  int V;
  int level;                 // position decided, in [0, K)
  int groups_per_slice;
  int num_groups;
};
cudaError_t level_prepare();
cudaError_t level_launch(const LevelArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                         cudaStream_t stream);

cudaError_t tile_tma_prepare(int max_smem_bytes);
int tile_tma_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes);
cudaError_t tile_tma_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid,
                            int smem_bytes, cudaStream_t stream);

cudaError_t tile_prepare(int max_smem_bytes);
int tile_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes);
cudaError_t tile_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid, int smem_bytes,
                        cudaStream_t stream);

}  // namespace specv
