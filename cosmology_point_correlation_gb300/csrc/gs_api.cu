// gs_api.cu -- small host entry points: configuration counts and indices, and
// the one-call host-buffer variants (copy in, build, count, copy out, free).

#include "gs_internal.cuh"

extern "C" int64_t gs_config_count_3pcf(int nbins)
{
    if (nbins < 1 || nbins > 255) return -1;
    return gs_ncfg3(nbins);
}

extern "C" int64_t gs_config_count_4pcf(int nbins)
{
    if (nbins < 1 || nbins > 255) return -1;
    return nbins < 3 ? 0 : gs_ncfg4(nbins);
}

extern "C" int64_t gs_config_index_3pcf(int nbins, int b1, int b2, int b3)
{
    if (nbins < 1 || nbins > 255 || b1 < 0 || b1 > b2 || b2 > b3 || b3 >= nbins) return -1;
    return gs_idx3(nbins, b1, b2, b3);
}

extern "C" int64_t gs_config_index_4pcf(int nbins, int b1, int b2, int b3)
{
    if (nbins < 3 || nbins > 255 || b1 < 0 || b1 >= b2 || b2 >= b3 || b3 >= nbins) return -1;
    return gs_idx4(nbins, b1, b2, b3);
}

extern "C" const char *gs_version(void)
{
    return GS_CHECKED_BUILD ? "gramsci_gb 0.2 (sm_103a, checked)" : "gramsci_gb 0.2 (sm_103a)";
}

// Copy host coordinates to the device and build the graph.
static gs_status build_from_host(const int32_t *coords_host, int64_t n, int64_t box_lu, int periodic,
                                 int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                                 cudaStream_t st, gs_graph_t *g)
{
    *g = nullptr;
    if (n > 0 && !coords_host) return gs_set_error(GS_ERR_ARG, "coords_host is NULL");
    int32_t *d = nullptr;
    if (n > 0) {
        GS_TRY_CUDA(gs_malloc_async(&d, sizeof(int32_t) * 3 * n, st));
        cudaError_t e = cudaMemcpyAsync(d, coords_host, sizeof(int32_t) * 3 * n, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) {
            cudaFreeAsync(d, st);
            return gs_set_error(GS_ERR_CUDA, "copy of coordinates failed: %s", cudaGetErrorString(e));
        }
    }
    gs_status s = gs_build_graph(d, n, box_lu, periodic, r_max_lu, edges_lu, nbins, st, g);
    if (d) cudaFreeAsync(d, st);
    return s;
}

extern "C" gs_status gs_3pcf_from_host(const int32_t *coords_host, int64_t n, int64_t box_lu, int periodic,
                                       int64_t r_max_lu, const int64_t *edges_lu, int nbins,
                                       uint64_t *hist_host, void *cuda_stream)
{
    GS_ENTRY();
    if (!hist_host) return gs_set_error(GS_ERR_ARG, "hist_host is NULL");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    gs_graph_t g = nullptr;
    gs_status s = build_from_host(coords_host, n, box_lu, periodic, r_max_lu, edges_lu, nbins, st, &g);
    if (s != GS_OK) return s;
    const int64_t ncfg = gs_ncfg3(nbins);
    uint64_t *h = nullptr;
    cudaError_t e = gs_malloc_async(&h, sizeof(uint64_t) * ncfg, st);
    if (e != cudaSuccess) {
        gs_graph_free(g);
        return gs_set_error(GS_ERR_NOMEM, "histogram allocation failed: %s", cudaGetErrorString(e));
    }
    s = gs_count_3pcf(g, h, 0, n, st);
    if (s == GS_OK) {
        e = cudaMemcpyAsync(hist_host, h, sizeof(uint64_t) * ncfg, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) s = gs_set_error(GS_ERR_CUDA, "histogram copy failed: %s", cudaGetErrorString(e));
    }
    cudaFreeAsync(h, st);
    gs_graph_free(g);
    return s;
}

extern "C" gs_status gs_4pcf_parity_from_host(const int32_t *coords_host, int64_t n, int64_t box_lu,
                                              int periodic, int64_t r_max_lu, const int64_t *edges_lu,
                                              int nbins, uint64_t *even_host, int64_t *odd_host,
                                              void *cuda_stream)
{
    GS_ENTRY();
    const int64_t ncfg = nbins >= 3 && nbins <= 255 ? gs_ncfg4(nbins) : 0;
    if (ncfg > 0 && (!even_host || !odd_host)) return gs_set_error(GS_ERR_ARG, "NULL histogram");
    cudaStream_t st = (cudaStream_t)cuda_stream;
    gs_graph_t g = nullptr;
    gs_status s = build_from_host(coords_host, n, box_lu, periodic, r_max_lu, edges_lu, nbins, st, &g);
    if (s != GS_OK) return s;
    if (ncfg == 0) {
        gs_graph_free(g);
        return GS_OK;
    }
    uint64_t *ev = nullptr;
    int64_t *od = nullptr;
    cudaError_t e = gs_malloc_async(&ev, sizeof(uint64_t) * ncfg, st);
    if (e == cudaSuccess) e = gs_malloc_async(&od, sizeof(int64_t) * ncfg, st);
    if (e != cudaSuccess) {
        if (ev) cudaFreeAsync(ev, st);
        gs_graph_free(g);
        return gs_set_error(GS_ERR_NOMEM, "histogram allocation failed: %s", cudaGetErrorString(e));
    }
    s = gs_count_4pcf_parity(g, ev, od, 0, n, st);
    if (s == GS_OK) {
        e = cudaMemcpyAsync(even_host, ev, sizeof(uint64_t) * ncfg, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(odd_host, od, sizeof(int64_t) * ncfg, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) s = gs_set_error(GS_ERR_CUDA, "histogram copy failed: %s", cudaGetErrorString(e));
    }
    cudaFreeAsync(ev, st);
    cudaFreeAsync(od, st);
    gs_graph_free(g);
    return s;
}
