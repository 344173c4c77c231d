// Instantiations of the pipelined chunk kernel for the per-token decay (the
// gate of the generic "decay, add, read out" loop of "Linear Attention, RWKV,
// and RetNet", 13.3 subsection 4); see chunk_tc_ws.cuh.  A translation unit of
// its own so that the two sets of instantiations compile in parallel.
#ifdef LA_TIMELINE
#undef LA_TIMELINE  // the development timeline lives in chunk_tc_ws.cu only
#endif
#include "chunk_tc_ws.cuh"

namespace la {

cudaError_t launch_chunk_tc_ws_gated(int dk, int dvb, bool normalize, const TcParams& prm,
                                     int grid, cudaStream_t s, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    return dispatch_ws<true>(dk, dvb, normalize, prm, grid, s, pdl);
}

}  // namespace la
