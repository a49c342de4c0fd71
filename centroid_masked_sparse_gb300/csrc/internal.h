// Host-side interface between the C ABI (mtp_head.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace mtp {

// Number of 256-element chunks a warp covers for rows of H bf16 values, rounded
// up to a compiled size; 0 if H is beyond the compiled sizes.
int chunks_for_hidden(int H);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Resident CTAs per SM for a kernel (cached per kernel and shared-memory size).
int blocks_per_sm(const void *kernel, int block, size_t smem);

// Raise a kernel's dynamic shared-memory limit once.
cudaError_t allow_smem(const void *kernel, size_t smem);

constexpr int kProjThreads = 256;
constexpr int kProjRowsPerWarp = 2;
constexpr int kTopkThreads = 256;
constexpr int kScoreThreads = 128;
constexpr int kScoreWarps = kScoreThreads / kWarp;

cudaError_t launch_projection(const ProjParams &p, cudaStream_t s);
cudaError_t launch_topk(const TopkParams &p, cudaStream_t s);
// Launches the persistent gather-score (or dense) kernel; *grid receives the CTA count.
cudaError_t launch_score(const ScoreParams &p, ScoreMode mode, cudaStream_t s, int *grid);
cudaError_t launch_fill_neg_inf(float *out, size_t n, cudaStream_t s);

}  // namespace mtp
