// Instantiations of the pipelined chunk kernel for the per-head decay gamma,
// and the dispatch for both decays (see chunk_tc_ws.cuh).
#include "chunk_tc_ws.cuh"

namespace la {

bool tc_ws_supported(int mode, int dk, int dvb, bool normalize) {
    if (opt_tc_lockstep()) return false;
    if (dk != 64 && dk != 128) return false;
    if (dvb != 64 && dvb != 128) return false;
    if (mode == kStateOnly) return true;
    if (mode != kFull) return false;
    return dvb == 64 || !normalize;
}

// Defined in chunk_tc_ws_gated.cu (the per-token decay's instantiations).
cudaError_t launch_chunk_tc_ws_gated(int dk, int dvb, bool normalize, const TcParams& prm,
                                     int grid, cudaStream_t s, bool pdl);

cudaError_t launch_chunk_tc_ws(int dk, int dvb, bool normalize, const TcParams& prm, int grid,
                               cudaStream_t s, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    if (prm.gate) return launch_chunk_tc_ws_gated(dk, dvb, normalize, prm, grid, s, pdl);
    return dispatch_ws<false>(dk, dvb, normalize, prm, grid, s, pdl);
}

}  // namespace la
