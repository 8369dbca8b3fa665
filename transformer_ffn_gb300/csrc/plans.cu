// plans.cu -- host-side views of the weight streams' work plans, for tests
// that need no GPU (declared in tffn.h).
#include "../../include/tffn.h"
#include "decode.cuh"
#include "wstream.cuh"

extern "C" int tffn_debug_stream_plan(int path, int64_t M, int64_t N, int64_t O, int64_t P, int sms, int glu,
                                      int64_t out[12])
{
    if (M < 1 || N < 1 || O < 1 || P < 1 || sms < 1 || out == nullptr)
        return TFFN_ERR_INVALID_ARG;
    if (path == 2) {
        const tffn::decode::Plan pl = tffn::decode::make_plan(M, N, O, P, sms, glu != 0);
        const int64_t v[12] = {pl.grid,      pl.win,       pl.nblk,      pl.slices[0], pl.slices[1], pl.kch[0],
                               pl.kch[1],    pl.units[0],  pl.units[1],  pl.maxp[0],   pl.maxp[1],
                               static_cast<int64_t>(pl.partial_bytes)};
        for (int i = 0; i < 12; ++i)
            out[i] = v[i];
        return TFFN_OK;
    }
    if (path == 6) {
        if (M > tffn::wstream::MAX_ROWS)
            return TFFN_ERR_UNSUPPORTED;
        const tffn::wstream::Plan pl = tffn::wstream::make_plan(M, N, O, P, sms, glu != 0);
        const int64_t v[12] = {pl.grid,      pl.win,       pl.nblk,      pl.slices[0], pl.slices[1], pl.kch[0],
                               pl.kch[1],    pl.units[0],  pl.units[1],  pl.maxp[0],   pl.maxp[1],
                               static_cast<int64_t>(pl.partial_bytes)};
        for (int i = 0; i < 12; ++i)
            out[i] = v[i];
        return TFFN_OK;
    }
    return TFFN_ERR_INVALID_ARG;
}
