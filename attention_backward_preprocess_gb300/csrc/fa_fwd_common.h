// fa_fwd_common.h -- what the two forward kernels share: the extension flags
// of an instance, the instances built, which of them give each query row two
// softmax warps, and the launcher of those.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_params.h"

namespace fa {

// Extension flags of a forward instance: ALiBi, the elementwise bias, dropout
// (the band needs none: only edge blocks test it).  Each extension gets
// compiled in only where asked for: its code slows the softmax even when
// skipped at run time.
enum : int { kFwdAlibi = 2, kFwdBias = 4, kFwdDrop = 8 };
// the instances built, each a superset of the flags before it in its chain
constexpr int kFwdFlagSets[] = {0, kFwdAlibi, kFwdAlibi | kFwdBias, kFwdDrop,
                                kFwdAlibi | kFwdBias | kFwdDrop};
constexpr int kNumFwdFlagSets = (int)(sizeof(kFwdFlagSets) / sizeof(int));

// The first instance built that has every flag needed.
constexpr int fwd_instance_flags(int need) {
    for (int i = 0; i < kNumFwdFlagSets; ++i)
        if ((need & kFwdFlagSets[i]) == need) return kFwdFlagSets[i];
    return kFwdFlagSets[kNumFwdFlagSets - 1];
}

// Instances whose softmax gives each query row two warps, each taking half of
// every block's keys (fa_fwd_split.cu): with the bias or dropout (more work per
// score) and at D = 64 (less MMA work to hide the softmax behind).  Measured on
// the 8k GQA workload, the plain and ALiBi instances at D = 128 run faster
// with one warp per row (fa_fwd_tc.cu): there the per-block exchange of the
// row maxima between the two warps costs more than the halved work saves.
constexpr bool fwd_split(int d, int flags) { return (flags & (kFwdBias | kFwdDrop)) != 0 || d == 64; }

// Launches the two-warps-per-row forward instance for (D, dtype, flags).
cudaError_t launch_fwd_split(const BwdParams &p, const CUtensorMap &q, const CUtensorMap &k,
                             const CUtensorMap &v, void *o, float *lse, int max_lq, int bf16,
                             int flags, cudaStream_t stream);

}  // namespace fa
