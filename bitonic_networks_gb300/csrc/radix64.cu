// radix64.cu -- the 64-bit key configuration of the LSD radix sort: 8 digit
// passes of radix 256 ([PMPP10] section 8, exercise 2), with the kernels of
// radix_kernels.cuh instantiated for 64-bit key words.  A tile holds 16 warps
// x 8 keys (4096 keys), so that keys [+ values] stay in registers at the same
// register budget as the 32-bit configuration.
#include "radix_kernels.cuh"

namespace gsort {

namespace {
using Keys64 = PassConfig<uint64_t, 16, 8, 3, kMatchTable>;    // keys only: three CTAs per SM
using Config64 = PassConfig<uint64_t, 16, 8, 2, kMatchTable>;  // pairs: two
using FreeConfig64 = FreePassConfig<uint64_t, 16, 8, 3>;       // the order-free first pass
static_assert(FreeConfig64::kTile == Config64::kTile && Keys64::kTile == Config64::kTile,
              "one tile size for every pass");
}

cudaError_t launch_pass_u64(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                            cudaStream_t s) {
    return pairs ? Config64::launch(a, pairs, xin, xout, tiles, s) : Keys64::launch_keys(a, pairs, xin, xout, tiles, s);
}

cudaError_t launch_pass_u64_free(const PassArgs &a, bool pairs, bool xin, bool xout, uint32_t tiles,
                                 cudaStream_t s) {
    return FreeConfig64::launch(a, pairs, xin, xout, tiles, s);
}

uint32_t pass_tile_u64() { return Config64::kTile; }

cudaError_t launch_hist_u64(const uint64_t *keys, uint32_t n, bool xf, uint64_t fmask, uint64_t flip,
                            int begin_bit, int passes, uint32_t last_mask, uint32_t *hist,
                            uint32_t *clear, uint32_t clear_words, cudaStream_t s, int sm_count,
                            const BinStartsOut &bs) {
    return launch_hist_kernel<uint64_t>(keys, n, xf, fmask, flip, begin_bit, passes, last_mask, hist,
                                        clear, clear_words, s, sm_count, bs);
}

}  // namespace gsort
