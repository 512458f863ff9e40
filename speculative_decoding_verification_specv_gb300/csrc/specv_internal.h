// specv_internal.h -- launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

constexpr int kRowThreads = 256;   // threads per CTA of the cluster row kernel
constexpr int kMaxCluster = 16;    // largest cluster (non-portable size, opt-in)
constexpr int kTileThreads = 256;  // threads per CTA of the small-vocabulary kernel
constexpr int kTmaTileLanes = 8;           // stage-B lanes per sequence of the TMA tile kernel
constexpr int kTmaTileMaxSeqs = kTileThreads / kTmaTileLanes;  // sequences per TMA tile (32)
constexpr int kResidentChunkGroups = 1024;  // 16-byte groups per TMA chunk (16 KiB per row)
constexpr int kResidentMaxChunks = 8;       // chunks per row slice (128 KiB per row at most)

// Sampler segments of the streaming row kernel.  A CTA's slice of a row is cut
// into segments of seg_tiles * kSegGroups consecutive 16-byte groups (the last
// one may be short), at most kMaxSegs per slice; a warp reads a tile of
// kSegGroups groups as kSegLaneGroups coalesced 16-byte loads per lane.
constexpr int kSegLaneGroups = 4;
constexpr int kSegGroups = 32 * kSegLaneGroups;
constexpr int kMaxSegs = 512;

// Segment geometry of a slice of groups_per_slice groups.
inline void rows_segments(int groups_per_slice, int *seg_tiles, int *segs_per_slice) {
  const int64_t tiles = ((int64_t)groups_per_slice + kSegGroups - 1) / kSegGroups;
  const int64_t per_seg = (tiles + kMaxSegs - 1) / kMaxSegs;
  *seg_tiles = (int)(per_seg < 1 ? 1 : per_seg);
  const int64_t seg_groups = (int64_t)*seg_tiles * kSegGroups;
  *segs_per_slice = (int)(((int64_t)groups_per_slice + seg_groups - 1) / seg_groups);
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
// staged = true: slices staged in shared memory by TMA; false: read in place
// from global memory (the sampler re-reads the slice, from L2 when it fits).
cudaError_t resident_launch(const ResArgs &a, int dtype_bf16, int mode, bool staged, int S,
                            int64_t grid, int smem, cudaStream_t stream);

cudaError_t rows_prepare();
cudaError_t rows_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                        int64_t grid, cudaStream_t stream);

cudaError_t tile_tma_prepare(int max_smem_bytes);
int tile_tma_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes);
cudaError_t tile_tma_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid,
                            int smem_bytes, cudaStream_t stream);

cudaError_t tile_prepare(int max_smem_bytes);
int tile_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes);
cudaError_t tile_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid, int smem_bytes,
                        cudaStream_t stream);

}  // namespace specv
