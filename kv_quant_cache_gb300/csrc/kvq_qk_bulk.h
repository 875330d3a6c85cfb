// kvq_qk_bulk.h -- internal interface of the TMA-staged QK kernel
// (kvq_qk_bulk.cu).  Not installed; callers use include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_launch.h"

namespace kvq {

// Staged launch shapes X(warps per CTA, stages per warp, rows per stage), in
// the order of their QK configuration entries (named bulk<Ww,Sst,Rr>).
#define KVQ_QK_BULK_SHAPES(X) X(16, 2, 24) X(24, 2, 12) X(24, 3, 8)
#define KVQ_QK_BULK_COUNT(W, S, R) +1
constexpr int kQkBulkShapes = 0 KVQ_QK_BULK_SHAPES(KVQ_QK_BULK_COUNT);

// True when staged shape `shape` may serve this call: the head_dim-128
// full-NeoX layout, qkv and the cos/sin table in device memory (the
// bulk-copy engine is not pointed at mapped host memory), and the token's
// rows split into non-empty chunks.
bool qk_bulk_eligible(const QkArgs& a, int shape);

// Launch staged shape `shape` (0 .. kQkBulkShapes-1) of the head_dim-128
// full-NeoX operator.
cudaError_t launch_qk_bulk(const QkArgs& a, int shape, cudaStream_t stream);

// Polls of a stage barrier after which a warp stops staging and finishes its
// items with direct loads (default 1 << 22).  Returns the previous value.
uint32_t set_qk_stage_wait_limit(uint32_t polls);

}  // namespace kvq
