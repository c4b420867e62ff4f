// Host-side construction of the synchronized channel set S.
//
// "Tensor-Parallelism with Partially Synchronized Activations": the partial
// channel-reduce sums "a subset of the channels" (Introduction); its size is the
// fraction p of the hidden dimension (experimental setup, p = 0.5).  Which
// channels form the subset is not stated; this library offers the leading block
// and a seeded uniform random subset.  The random subset comes from a
// Fisher-Yates shuffle driven by SplitMix64 (Steele, Lea & Flood, OOPSLA 2014),
// so any implementation of that published generator reproduces it.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "caat.h"

namespace {

struct SplitMix64 {
    uint64_t state;
    uint64_t next()
    {
        state += 0x9e3779b97f4a7c15ULL;             // golden-ratio increment
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL; // Stafford mix13
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
        return z ^ (z >> 31);
    }
};

}  // namespace

extern "C" caat_status caat_select_channels(int64_t h, double p, caat_layout layout,
                                            uint64_t seed, int32_t *idx, int64_t *n_sel)
{
    if (h < 0 || h > INT32_MAX || !(p >= 0.0 && p <= 1.0) || n_sel == nullptr)
        return CAAT_ERR_INVALID_ARG;
    if (layout != CAAT_S_CONTIGUOUS && layout != CAAT_S_RANDOM) return CAAT_ERR_INVALID_ARG;
    if (idx == nullptr && h > 0) return CAAT_ERR_INVALID_ARG;
    int64_t s = (int64_t)std::floor(p * (double)h + 0.5);
    s = std::min<int64_t>(std::max<int64_t>(s, 0), h);
    if (layout == CAAT_S_CONTIGUOUS) {
        for (int64_t i = 0; i < s; ++i) idx[i] = (int32_t)i;
    } else {
        std::vector<int32_t> pi((size_t)h);
        for (int64_t i = 0; i < h; ++i) pi[(size_t)i] = (int32_t)i;
        SplitMix64 g{seed};
        for (int64_t i = h - 1; i >= 1; --i) {
            const uint64_t j = g.next() % (uint64_t)(i + 1);
            std::swap(pi[(size_t)i], pi[(size_t)j]);
        }
        std::sort(pi.begin(), pi.begin() + s);
        std::copy(pi.begin(), pi.begin() + s, idx);
    }
    *n_sel = s;
    return CAAT_OK;
}
