// grouped_sched.cuh -- group resolution and tile order shared by the grouped kernels.
//
// Every CTA reads m_sizes (int64, device memory), checks it (no negative entry, sum ==
// total_M) and prefix-sums it into a shared-memory table; a flat tile id then maps to
// (group, 128-row block of that group, column block).  Empty groups own no tiles, no
// tile spans two groups, and rows past a group's end are computed but never stored
// ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm": the commit that replaced the host
// tile map by in-kernel group resolution; "PyTorch on AMD GPUs gains a FlyDSL backend",
// Interpretation: uneven and empty expert groups).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace bsmma {
namespace grouped {

constexpr int kBM = 128;    // rows of a tile
constexpr int kMaxG = 64;   // groups per launch

struct GroupTable {
  int64_t start[kMaxG + 1];   // first row of each group
  int64_t size[kMaxG];
  int tile_start[kMaxG + 1];  // first row-block id of each group
  int bad;
};

// Fills `gt` from m_sizes, counting row blocks of TR rows; called by every thread of the
// block (needs blockDim >= G).  A bad table latches kDevBadMSizes once (block 0) and sets
// gt.bad for every block.  `init` runs on thread 0 between the table and the closing
// barrier (barrier setup).
template <int TR = kBM, typename Init>
__device__ __forceinline__ void build_group_table(GroupTable& gt, const int64_t* m_sizes, int G,
                                                  int64_t total_M, int* status, Init init) {
  if (threadIdx.x < G) gt.size[threadIdx.x] = m_sizes[threadIdx.x];
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t row = 0;
    int tiles = 0, bad = 0;
    for (int g = 0; g < G; ++g) {
      const int64_t m = gt.size[g];
      if (m < 0 || m > total_M) bad = 1;
      gt.start[g] = row;
      gt.tile_start[g] = tiles;
      if (!bad) {
        row += m;
        tiles += static_cast<int>((m + TR - 1) / TR);
      }
    }
    if (row != total_M) bad = 1;
    gt.start[G] = row;
    gt.tile_start[G] = tiles;
    gt.bad = bad;
    if (bad && blockIdx.x == 0) report_status(status, kDevBadMSizes);
    init();
  }
  __syncthreads();
}

// Tile t -> (row block mt, column block nt).  Tiles are walked in bands of kBandRows
// row blocks: within a band the row block varies fastest, so the CTAs resident at one
// time share a few weight column blocks and a band's rows of X, both of which stay in
// L2 while the band is walked along N (row-fastest over all rows re-read every group's
// whole weight matrix from DRAM for every few row blocks).
constexpr int kBandRows = 16;
__device__ __forceinline__ void tile_coords(int t, int NT, int rows, int& mt, int& nt) {
  const int per_band = kBandRows * NT;
  const int b = t / per_band;
  const int r0 = b * kBandRows;
  const int h = rows - r0 < kBandRows ? rows - r0 : kBandRows;
  const int v = t - b * per_band;
  mt = r0 + v % h;
  nt = v / h;
}

// Group owning row block `mt` (tile_start is non-decreasing; empty groups own none).
__device__ __forceinline__ int find_group(const GroupTable& gt, int G, int mt) {
  int g = 0;
  for (int i = 1; i < G; ++i)
    if (gt.tile_start[i] <= mt) g = i;
  return g;
}

}  // namespace grouped
}  // namespace bsmma
