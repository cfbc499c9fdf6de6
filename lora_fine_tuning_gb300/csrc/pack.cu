// Greedy token-capacity packing of samples into microbatches (host only).
//
// The multi-adapter scheduler of the LoRAFusion pages (notes on
// papers.chlience.com, section 5 "Multi-LoRA scheduler"; the juhe.plus
// article, section 4.2 step 2) fills microbatches up to a token capacity with
// a two-stage MILP and falls back to greedy packing when the solver runs out
// of time.  This is that greedy: first-fit decreasing, where a sample takes
// its length rounded up to whole 128-row tiles (the unit the multi-adapter
// kernels route).  The result feeds multi_lora_fwd / multi_lora_bwd: the
// samples of microbatch b, at their rows, are its segment table.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "lora.h"

extern "C" lora_status lora_pack_greedy(const int64_t* lengths, int32_t n_samples, int64_t capacity,
                                        int32_t* batch_of_sample, int64_t* row_of_sample, int32_t* n_batches) {
    if (n_samples < 0 || !n_batches || (n_samples > 0 && (!lengths || !batch_of_sample || !row_of_sample)))
        return LORA_EINVAL;
    if (capacity <= 0 || capacity % LORA_TILE_ROWS) return LORA_EINVAL;
    std::vector<int64_t> size(static_cast<size_t>(n_samples));
    for (int32_t i = 0; i < n_samples; ++i) {
        if (lengths[i] < 1) return LORA_EINVAL;
        size[i] = (lengths[i] + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS * LORA_TILE_ROWS;
        if (size[i] > capacity) return LORA_ESHAPE;
    }
    // longest first; equal sizes keep sample order
    std::vector<int32_t> order(static_cast<size_t>(n_samples));
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return size[a] > size[b]; });
    std::vector<int64_t> used;   // rows filled in each microbatch, in opening order
    for (const int32_t i : order) {
        size_t b = 0;
        while (b < used.size() && used[b] + size[i] > capacity) ++b;
        if (b == used.size()) used.push_back(0);
        batch_of_sample[i] = static_cast<int32_t>(b);
        row_of_sample[i] = used[b];
        used[b] += size[i];
    }
    *n_batches = static_cast<int32_t>(used.size());
    return LORA_OK;
}
