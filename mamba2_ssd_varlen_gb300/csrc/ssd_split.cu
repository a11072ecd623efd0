// ssd_split.cu -- block-aligned prefill bites, host side ("Automatic prefix
// caching for GDN hybrid models (mamba_cache_mode=all) with MTP speculative
// decoding", Purpose, the engine-core bullet: kernel-chunk-aligned prefill
// clipping and block-aligned split in the scheduler; and the review note on
// that page: a misaligned start is re-aligned at the next boundary even in the
// final bite, after which the last bite may end anywhere).
//
// A scheduler that prefills a long prompt in bites under a token budget asks
// here where a proposed bite [start, end) should end so that each later bite
// starts on the align grid (the block size, a multiple of the chunk size).
// The forward cuts chunks at absolute positions, so block checkpoints are exact
// for any bite; aligned bites additionally make every bite's end state a block
// checkpoint and keep bites from splitting a block between steps.
#include "ssd_internal.cuh"

extern "C" int64_t ssd_varlen_align_bite(int64_t start, int64_t end, int64_t total, int32_t align) {
    if (align < 1 || start < 0 || end <= start || end > total) return SSD_ERR_DIMS;
    const int64_t last_aligned = total / align * align;  // the last boundary inside the prompt
    if (start % align != 0) {
        // re-align a misaligned start (e.g. a prefix computed elsewhere) at the
        // next boundary, when the prompt reaches it, even in the final bite
        const int64_t next = (start / align + 1) * align;
        return next <= last_aligned ? (end < next ? end : next) : end;
    }
    // An aligned bite that stops short of the last boundary ends on a boundary;
    // a budget below one block gives start (nothing this step).
    if (end < last_aligned) return end / align * align;
    return end;  // an aligned start reaching the last boundary: the prompt's tail may end anywhere
}
