// kvq_qk_bulk.h -- internal interface of the TMA-staged QK kernel
// (kvq_qk_bulk.cu).  Not installed; callers use include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_launch.h"

namespace kvq {

// Staged launch shapes X(warps per CTA, stages per warp, KB of head rows per
// stage, tiled), in the order of their QK configuration entries (named
// bulk<Ww,Sst,KKB> and, for tiled tensor-map copies, bulk<Ww,Sst,KKB,tile>).
// A stage holds KB * 1024 / (2 head_dim) rows plus one cos/sin row.
#define KVQ_QK_BULK_SHAPES(X) X(16, 2, 6, 0) X(24, 2, 3, 0) X(24, 3, 2, 0) X(16, 2, 6, 1)
#define KVQ_QK_BULK_COUNT(W, S, KB, T) +1
constexpr int kQkBulkShapes = 0 KVQ_QK_BULK_SHAPES(KVQ_QK_BULK_COUNT);
// Index of the first staged shape in the QK configuration table.
constexpr int kQkFirstBulk = 7;

// True when staged shape `shape` may serve this call: a supported head_dim,
// qkv and the cos/sin table in device memory (the bulk-copy engine is not
// pointed at mapped host memory), and the token's rows split into non-empty
// chunks.
bool qk_bulk_eligible(const QkArgs& a, int shape);

// Launch staged shape `shape` (0 .. kQkBulkShapes-1) for any supported
// layout (head_dim 64 / 128 / 256, NeoX or GPT-J, full or partial rotation).
cudaError_t launch_qk_bulk(const QkArgs& a, int shape, cudaStream_t stream);

// The staging-event counters of the current device (kvq_stage_events):
// waits for the device to finish its work, reads [fallbacks, drain
// timeouts] and zeroes them if `reset`.
cudaError_t stage_events(uint64_t out[2], bool reset);

}  // namespace kvq
