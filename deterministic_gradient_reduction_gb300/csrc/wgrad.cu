// Split-K grouped weight gradient accumulated into fp32 main_grad.
#include "dgr_common.cuh"

using namespace dgr;

extern "C" size_t dgr_wgrad_workspace_bytes(int32_t E, int64_t N, int64_t K) {
    (void)E;
    (void)N;
    (void)K;
    return sizeof(WsHeader);
}

extern "C" dgr_status dgr_grouped_wgrad_accumulate(const void *G, const void *X, const int64_t *d_offs,
                                                   int32_t E, int64_t T_total, int64_t N, int64_t K,
                                                   float *main_grad, int32_t chunk_tokens, void *ws,
                                                   size_t ws_bytes, void *stream) {
    (void)G; (void)X; (void)d_offs; (void)E; (void)T_total; (void)N; (void)K; (void)main_grad;
    (void)chunk_tokens; (void)ws; (void)ws_bytes; (void)stream;
    return DGR_ERR_UNSUPPORTED;
}
