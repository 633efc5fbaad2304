// Test aid: the host-side planner of the C ABI -- the tile cost model, the
// cluster shape, the stream-K schedule and its cut table, an operand's byte
// extent and whether a tensor map can read it -- exposed with C
// linkage so that CPU tests can call it with a GPU's resource counts (SMs,
// resident clusters) given as numbers.  The library's host source is compiled
// into this test library as it stands; the kernel launchers it refers to come
// from libgemm_gb300.so, which this library links against, and no test calls
// them.
#include "../dense_gemm_epilogues_tcgen05_gb300/csrc/gemm_api.cu"

extern "C" {

// Tile family (1: one SM per 128 x bn tile, 2: an SM pair per 256 x bn tile); *bn gets the width.
int plan_choose_tile(int64_t M, int64_t N, int num_sms, int max_clusters, int policy, int policy_bn, int *bn) {
    const TileChoice t = choose_tile(M, N, num_sms, max_clusters, policy, policy_bn);
    *bn = t.bn;
    return t.kind;
}

// CTAs per cluster of the pair kernel (2 or 4).
int plan_choose_cluster(int64_t tiles, int64_t tiles_n, int max_pairs, int max_quads, int a_splits, int mode) {
    return choose_cluster(tiles, tiles_n, max_pairs, max_quads, a_splits != 0, mode);
}

// Schedule of `tiles` units of `num_kb` k-blocks over at most `max_clusters`
// clusters; cuts must hold kMaxSkClusters + 1 entries.
void plan_choose_schedule(int64_t tiles, int num_kb, int max_clusters, int have_ws, int mode, int bn, int *dp_tiles,
                          long long *sk_units, unsigned int *cuts, int *clusters) {
    choose_schedule(tiles, num_kb, max_clusters, have_ws != 0, mode, bn, dp_tiles, sk_units, cuts, clusters);
}

// The cut table (clusters + 1 entries) and the feasibility test it is searched with.
void plan_stream_k_cuts(long long units, int num_kb, int clusters, int dp_tiles, long long e_kb,
                        unsigned int *cuts) {
    stream_k_cuts(units, num_kb, clusters, dp_tiles, e_kb, cuts);
}

int plan_stream_k_feasible(long long units, int num_kb, int clusters, int dp_tiles, long long e_kb, long long limit,
                           unsigned int *cuts) {
    return stream_k_feasible(units, num_kb, clusters, dp_tiles, e_kb, limit, cuts) ? 1 : 0;
}

int plan_max_sk_clusters() { return kMaxSkClusters; }

// Bytes from an operand's first element to one past its last (the range checked against its allocation).
unsigned long long plan_span_bytes(int64_t rows, int64_t cols, int64_t s_rows, int64_t s_cols, int es) {
    return span_bytes(rows, cols, s_rows, s_cols, es);
}

// How an (mn x k) operand at address `base` is read: 0 no tensor map (CUDA-core path), 1 by a
// K-contiguous map, 2 by an MN-contiguous map.  The address is only tested for alignment.
int plan_operand_kind(unsigned long long base, int64_t mn, int64_t k, int64_t s_mn, int64_t s_k, int es) {
    const Operand o = plan_operand(reinterpret_cast<const void *>(base), mn, k, s_mn, s_k, es);
    return !o.tma ? 0 : (o.mn_major ? 2 : 1);
}

}  // extern "C"
