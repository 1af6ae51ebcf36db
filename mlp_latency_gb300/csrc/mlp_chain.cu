// mlp_chain.cu -- C ABI of the CTA-pipelined GEMM chain (see include/mlp_chain.h): handle
// creation, TMA descriptor encoding, and the three launch modes (pipelined, sequential,
// micro-batched) of the one tile engine in chain_kernel.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/mlp_chain.h"
#include "chain_kernel.cuh"
#include "dep_groups.h"

using mlpc::ChainParams;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 tensor map over a rows x cols row-major matrix, box = box_rows x box_cols.
bool encode_2d(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int box_rows, int box_cols,
               CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand map over K x N row-major weights, in boxes of k_rows x (b_swz / 2) columns.  When N
// is a multiple of the box width the map is a 3-D view (column in box, k, box) with the box
// stride one box row (b_swz bytes): one copy then loads all BN / box columns of a tile in the
// same shared-memory layout as one 2-D copy per box, with a single instruction to issue.  A
// ragged N keeps the 2-D map, whose bounds zero-fill the columns past N.
bool encode_w_kn(CUtensorMap *map, const void *ptr, int64_t K, int64_t N, int k_rows, int b_swz, int bn,
                 int32_t *is_3d)
{
    const int box_cols = b_swz / 2;
    const CUtensorMapSwizzle swz = b_swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    *is_3d = 0;
    if (bn <= box_cols || N % box_cols != 0 || bn % box_cols != 0)   // (tiles must start on a box)
        return encode_2d(map, ptr, K, N, k_rows, box_cols, swz);
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(box_cols), static_cast<cuuint64_t>(K),
                          static_cast<cuuint64_t>(N / box_cols)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(b_swz)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(k_rows),
                         static_cast<cuuint32_t>(bn / box_cols)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return encode_2d(map, ptr, K, N, k_rows, box_cols, swz);   // the driver refused the view
    *is_3d = 1;
    return true;
}

// Views whose outermost coordinate is the 64-deep k block, for fills of two k blocks: one copy
// then lands both blocks' tiles one after the other, each in the layout of a one-block copy.
//   activations (rows x K, row-major), or weights stored N x K: (k in block, row, k block);
//   weights stored K x N: (column in box, k in block, box, k block).
bool encode_kblocks(CUtensorMap *map, const void *ptr, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void *>(ptr), dims,
              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_kblocks(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K, int box_rows)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(mlpc::kBK), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(K / mlpc::kBK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(mlpc::kBK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(mlpc::kBK), static_cast<cuuint32_t>(box_rows), 2};
    return encode_kblocks(map, ptr, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_w_kn_kblocks(CUtensorMap *map, const void *ptr, int64_t K, int64_t N, int b_swz, int bn)
{
    const int box_cols = b_swz / 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(box_cols), static_cast<cuuint64_t>(mlpc::kBK),
                                static_cast<cuuint64_t>(N / box_cols), static_cast<cuuint64_t>(K / mlpc::kBK)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(b_swz),
                                   static_cast<cuuint64_t>(N) * 2 * mlpc::kBK};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(mlpc::kBK),
                               static_cast<cuuint32_t>(bn / box_cols), 2};
    return encode_kblocks(map, ptr, 4, dims, strides, box,
                          b_swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

struct DeviceBoundary {
    int32_t *pg_off = nullptr, *pg_tgt = nullptr, *grp_off = nullptr, *grp_mem = nullptr, *grp_init = nullptr;
    int32_t *cgrp = nullptr;
    uint32_t *count = nullptr, *tail = nullptr, *ready = nullptr;
    unsigned long long *queue = nullptr;
    size_t groups = 0, consumers = 0, producers = 0;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// First-stage raster (and consumer grouping) when the caller leaves it to the library: groups of
// 8 row panels from 16 panels up, of 4 from 8 (measured best on GB300 for 16 and 64 panels; a
// group of all panels serialises the stages).  Below 8 panels, one group of all of them when the
// first stage takes more than one wave of cluster items: a later wave then reads each weight slab
// together with the other panels' tiles instead of re-reading the slabs an earlier wave streamed
// (SwiGLU MLP, 2 panels: 126 -> 103 us; 3, 4 and 6 panels of 256 rows at d = 8192: 5-7 %
// faster); a single wave reads every slab together in either order (Llama MLP: 77 us row by
// row against 78 grouped).
int default_raster_group(int tiles_m, int first_stage_items, int clusters)
{
    if (tiles_m >= 16)
        return 8;
    if (tiles_m >= 8)
        return 4;
    return first_stage_items > clusters ? tiles_m : 1;
}

// Both pipelined modes run one persistent, co-resident grid over all stages.
bool is_pipelined(int mode)
{
    return mode == MLP_MODE_PIPELINED || mode == MLP_MODE_PIPELINED_KWAIT || mode == MLP_MODE_PIPELINED_LAMPORT;
}

// Lamport runs: every intermediate starts as the sentinel, bf16 -0.0 (two per 32-bit word).
__global__ void fill_sentinel_kernel(uint4 *p, size_t n16)
{
    const uint4 v = make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

}  // namespace

struct mlp_chain {
    mlp_chain_desc desc{};
    int device = 0, num_sms = 0, S = 0;
    int bm = mlpc::kBM;      // rows per CTA's tile: 128, or 64 (tcgen05 M = 64)
    int pair = 1;            // 2: CTA pairs, each tile pair x bm rows (chain_kernel<2>)
    int raster_group = 1;    // first-stage raster and consumer grouping (row panels per group)
    int BN[MLP_MAX_GEMMS] = {}, tiles_m = 0, tiles_n[MLP_MAX_GEMMS] = {}, k_blocks[MLP_MAX_GEMMS] = {};
    int b_swz[MLP_MAX_GEMMS] = {};
    int num_pipe = 0, max_bn = 0, grid = 0, acc_split = 1;
    size_t meta_bytes = 0;   // bytes from d_ctrl through the last boundary's tables
    int cs = 1, max_clusters = 0;
    uint32_t recv_bytes = 0;
    int split[MLP_MAX_GEMMS] = {}, kb_per_split[MLP_MAX_GEMMS] = {}, items[MLP_MAX_GEMMS] = {};
    int kpf[MLP_MAX_GEMMS] = {};   // 64-deep k blocks per ring fill (1 or 2)
    bool xsplit[MLP_MAX_GEMMS] = {};   // k-slices on separate clusters (StageParams::xsplit)
    uint32_t *xcount[MLP_MAX_GEMMS] = {};
    int32_t tile_base[MLP_MAX_GEMMS + 1] = {};
    float *partials[MLP_MAX_GEMMS] = {};
    uint32_t stage_bytes = 0, tmem_cols = 0;
    size_t smem = 0;
    std::vector<int32_t> off[MLP_MAX_GEMMS - 1], tgt[MLP_MAX_GEMMS - 1], init[MLP_MAX_GEMMS - 1];
    mlpc::DepGroups grp[MLP_MAX_GEMMS - 1];
    void *dev_block = nullptr;
    DeviceBoundary db[MLP_MAX_GEMMS - 1];
    uint32_t *d_ctrl = nullptr;  // words: 0 ticket, 1 status, 2 seq, 4-5 launch counter (u64)
    mlpc::EventRec *d_events = nullptr;
    size_t n_events = 0;
    int32_t stage_base[MLP_MAX_GEMMS + 1] = {};
    // cached launch parameters (tensor maps are re-encoded only when a pointer changes)
    ChainParams params;
    const void *c_X = nullptr, *c_W[MLP_MAX_GEMMS + 1] = {}, *c_Y = nullptr, *c_ws = nullptr;
    int n_w = 0;             // weight pointers per run: S, plus the up matrix of a gated chain
    int acc_cols = 0;        // TMEM columns of one accumulator buffer
    bool params_valid = false;
    bool fault_armed = false;   // MLP_DEBUG_DROP_DECREMENT fires on the first run only
    // micro-batch streams and events
    cudaStream_t side[MLP_MAX_GEMMS] = {};
    std::vector<cudaEvent_t> events;
    cudaEvent_t fork = nullptr;
    int n_chunks = 0, chunk_tiles = 0;
};

extern "C" const char *mlp_status_str(mlp_status s)
{
    switch (s) {
    case MLP_OK: return "ok";
    case MLP_ERR_INVALID_ARG: return "invalid argument";
    case MLP_ERR_UNSUPPORTED: return "unsupported";
    case MLP_ERR_CUDA: return "CUDA error";
    case MLP_ERR_OOM: return "out of device memory";
    case MLP_ERR_TIMEOUT: return "bounded device wait timed out";
    case MLP_ERR_DEVICE_STATE: return "device state needs a reset";
    case MLP_ERR_BAD_TILE: return "dequeued tile id out of range";
    }
    return "unknown status";
}

// Tile width and split-K factor of one stage, from a cost model of this kernel on one SM:
// one tcgen05.mma (M = 128, K = 16) costs about the same for any N <= 256 (~140 cycles), a TMA
// box row (64 or 128 bytes) costs ~1.2 ns, a split tile pays ~4 us for its fp32 reduction,
// and a stage cannot beat the HBM time of its weights.  With CTA pairs (pair = 2) a tile is
// 2 bm rows on two SMs, each loading bm activation rows and half of the weight tile; a k-slice
// of a split tile then takes a pair, and a cluster holds pair x S CTAs.  tiles_m counts row
// tiles of pair x bm rows; clusters[i] = co-resident clusters of 2^i CTAs.  Candidates with
// idle k slices or reduction slices narrower than 32 columns are skipped.  Two bounds on a k
// block that the plain rate misses, used when comparing whole plans: the ring's depth
// (`ring_slots` fills of ~1.8 us round trip in flight) and `kb_floor`, the per-k-block cost of a
// 256-wide pair tile (~0.33 us measured).  Widths that are not powers of two (96 to 224 columns:
// their last 64-column box of weights is loaded whole, one copy per box) run only where asked
// for: 224-wide pair tiles put the GeLU chain's 74 tiles on 76 pairs instead of 64, and still
// measured slower (216 against 203 us; the 2-GEMM chain at M = 512: 108 against 101 us), the
// extra copies per k block costing more than the smaller MMAs save.  Returns the estimated
// microseconds.
static double choose_tiles(int64_t tiles_m, int bm, int64_t K, int64_t N, const int clusters[4], int fixed_bn,
                           int fixed_split, int *bn_out, int *split_out, int pair = 1, int ring_slots = 0,
                           double kb_floor = 0.0, bool split_one_wave = false)
{
    const int k_blocks = static_cast<int>((K + 63) / 64);
    double best = 1e30;
    *bn_out = 256;
    *split_out = 1;
    const int bns[8] = {256, 224, 192, 160, 128, 96, 64, 32};
    for (int bn : bns) {
        const bool pow2 = (bn & (bn - 1)) == 0;
        if (fixed_bn && bn != fixed_bn)
            continue;
        if (pair == 2 && bn < 128)   // a pair's CTA loads at least 64 weight columns
            continue;
        if (!pow2 && !fixed_bn)
            continue;
        if (!fixed_bn && bn < 128 && N > bn)   // narrow tiles only to cover narrow outputs
            continue;
        if (!fixed_bn && bn > 32 && N <= bn / 2)
            continue;
        for (int li = 0; li + (pair == 2 ? 1 : 0) < 4; ++li) {
            const int S = 1 << li;
            const int ci = li + (pair == 2 ? 1 : 0);   // cluster of pair x S CTAs
            if (fixed_split && S != fixed_split)
                continue;
            const int kbps = (k_blocks + S - 1) / S;
            if (bn / S < 32 || bn % S || (bn / S) % 32 || (S - 1) * kbps >= k_blocks || clusters[ci] < 1)
                continue;
            const double tiles = static_cast<double>(tiles_m) * ((N + bn - 1) / bn);
            const double cap = static_cast<double>(clusters[ci]) * S * pair;   // CTAs resident at once
            const double units = tiles * S * pair;
            if (split_one_wave && S > 1 && units > cap)   // slices on separate clusters: one wave only
                continue;
            // a persistent grid quantises into whole waves only while units are few
            const double waves = units <= 2 * cap ? std::ceil(units / cap) : units / cap;
            const int b_cols = (bn / pair + 63) / 64 * 64;   // weight columns one CTA loads per k block
            const double rows = bm + (bn / pair >= 64 ? b_cols : 64);
            // measured on GB300: a 128 x N x 16 MMA takes about max(48, N / 2) cycles; the
            // streaming rate with the MMAs running is about 1.2 ns per 128-byte operand row
            const double t_mma = kbps * 4 * std::max(48.0, bn / 2.0) / 2000.0;   // us
            const double t_tma = kbps * rows * 1.2e-3;                           // us
            const double t_lat = kbps * std::max(kb_floor, ring_slots ? 1.8 / ring_slots : 0.0);
            // a split tile's exchange: ~4 us in a cluster; slices on separate clusters exchange through
            // a gpu-scope fence, counter and acquire, measured ~3 us more per split stage (M = 256,
            // two 4096^2 GEMMs split four ways: 45.6 against 43.5 us for one CTA per tile)
            const double t_split = S > 1 ? (split_one_wave ? 7.0 : 4.0) : 0.0;
            const double t_unit = std::max(std::max(t_mma, t_tma), t_lat) + 1.0 + t_split;
            const double t_hbm = static_cast<double>(K) * N * 2 / 6.5e6;
            const double t = std::max(waves * t_unit, t_hbm);
            if (t < best * 0.999) {
                best = t;
                *bn_out = bn;
                *split_out = S;
            }
        }
    }
    return best;
}

// Scoreboard releases one producer tile of stage b makes per run: one per epilogue warp of each
// CTA of the tile (each split-K slice, each CTA of a pair).
static int releases_per_tile(const mlp_chain *h, int b)
{
    return h->pair * h->split[b] * mlpc::kEpiWarps;
}

static mlp_status full_reset(mlp_chain *h)
{
    if (cudaSetDevice(h->device) != cudaSuccess)
        return MLP_ERR_CUDA;
    if (cudaMemset(h->d_ctrl, 0, 8 * sizeof(uint32_t)) != cudaSuccess)
        return MLP_ERR_CUDA;
    for (int b = 0; b + 1 < h->S; ++b) {
        const DeviceBoundary &db = h->db[b];
        if (cudaMemset(db.count, 0, db.groups * sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(db.queue, 0, db.consumers * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMemset(h->db[b].tail, 0, sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(db.ready, 0, db.producers * sizeof(uint32_t)) != cudaSuccess)
            return MLP_ERR_CUDA;
    }
    for (int s = 0; s < h->S; ++s)
        if (h->xcount[s] &&
            cudaMemset(h->xcount[s], 0, static_cast<size_t>(h->tiles_m) * h->tiles_n[s] * h->pair * 4) != cudaSuccess)
            return MLP_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? MLP_OK : MLP_ERR_CUDA;
}

static void release(mlp_chain *h)
{
    if (!h)
        return;
    cudaSetDevice(h->device);
    for (auto &e : h->events)
        if (e)
            cudaEventDestroy(e);
    if (h->fork)
        cudaEventDestroy(h->fork);
    for (auto &s : h->side)
        if (s)
            cudaStreamDestroy(s);
    if (h->dev_block)
        cudaFree(h->dev_block);
    delete h;
}

extern "C" mlp_status mlp_chain_create(const mlp_chain_desc *d, mlp_chain_t *out)
{
    if (!d || !out)
        return MLP_ERR_INVALID_ARG;
    *out = nullptr;
    const int S = d->num_gemms;
    if (S < 1 || S > MLP_MAX_GEMMS || d->M < 1 || d->M > (int64_t)1 << 30)
        return MLP_ERR_INVALID_ARG;
    for (int s = 0; s <= S; ++s)
        if (d->dims[s] < 8 || d->dims[s] % 8 != 0 || d->dims[s] > (int64_t)1 << 24)
            return MLP_ERR_INVALID_ARG;
    if (d->in_dtype != MLP_DT_BF16 || d->acc_dtype != MLP_DT_F32 || d->h_dtype != MLP_DT_BF16 ||
        d->out_dtype != MLP_DT_BF16)
        return MLP_ERR_UNSUPPORTED;
    if (!(d->tile_m == 0 || d->tile_m == 64 || d->tile_m == 128) ||
        !(d->tile_k == 0 || d->tile_k == 64 || d->tile_k == 128))
        return MLP_ERR_UNSUPPORTED;
    if (d->epilogue != MLP_EPI_NONE && d->epilogue != MLP_EPI_GELU_TANH)
        return MLP_ERR_INVALID_ARG;
    if (d->residual && d->dims[S] != d->dims[0])
        return MLP_ERR_INVALID_ARG;
    if (!is_pipelined(d->mode) && d->mode != MLP_MODE_SEQUENTIAL && d->mode != MLP_MODE_MICROBATCH &&
        d->mode != MLP_MODE_SEQUENTIAL_PDL)
        return MLP_ERR_INVALID_ARG;
    const int bm = d->tile_m == 64 ? 64 : mlpc::kBM;
    if (d->cta_pair < 0 || d->cta_pair > 2)
        return MLP_ERR_INVALID_ARG;
    // CTA pairs run no split accumulators, 64-row tiles, K-granular or Lamport modes or
    // shared-memory split-K exchange; tiles 128 or 256 wide (64 or 128 columns per CTA), a gated
    // GEMM's 64 or 128 wide (one CTA loads the gate tile, the other the up tile)
    bool pair_ok = d->acc_split != 2 && d->tile_m != 64 && d->mode != MLP_MODE_PIPELINED_KWAIT &&
                   d->mode != MLP_MODE_PIPELINED_LAMPORT && d->splitk_exchange != 2 && d->tile_k != 128;
    // Fills of two k blocks: one CTA per tile, one accumulator, and no per-k-block consumer work
    // (the K-granular waits and the Lamport scan are per 64-deep block)
    const bool deep_ok = d->acc_split != 2 && d->mode != MLP_MODE_PIPELINED_KWAIT && d->mode != MLP_MODE_PIPELINED_LAMPORT;
    if (d->tile_k == 128 && (!deep_ok || d->cta_pair == 2))
        return MLP_ERR_UNSUPPORTED;
    for (int s = 0; s < S && pair_ok; ++s)
        pair_ok = d->tile_n[s] == 0 || d->tile_n[s] >= (d->gated && s == 0 ? 64 : 128);
    if (d->cta_pair == 2 && !pair_ok)
        return MLP_ERR_UNSUPPORTED;
    if (d->mode == MLP_MODE_MICROBATCH && (d->microbatch_rows < bm || d->microbatch_rows % bm ||
                                           (d->cta_pair == 2 && d->microbatch_rows % (2 * bm))))
        return MLP_ERR_INVALID_ARG;
    // the library does not choose pairs for micro-batching: with concurrent chunk launches they
    // measured slower on the GeLU chain (256-row chunks: 462 against 332 us) and faster on prefill
    // (1024-row chunks: 384 against 441 us), so they stay an explicit option there
    const bool pair_auto_ok = pair_ok && d->mode != MLP_MODE_MICROBATCH;
    if (d->gated && (d->acc_split == 2 || (d->tile_n[0] != 0 && d->tile_n[0] > 128) ||
                     (d->k_split[0] != 0 && d->k_split[0] != 1)))
        return MLP_ERR_UNSUPPORTED;   // the gated GEMM keeps gate and up side by side in TMEM, unsplit
    if (d->grid_ctas < 0 || d->raster_group < 0 || d->pipe_stages < 0 || d->pipe_stages == 1 ||
        d->pipe_stages > mlpc::kMaxPipe || d->acc_split < 0 || d->acc_split > 2 || d->weight_layout < 0 ||
        d->weight_layout > 1 || d->splitk_exchange < 0 || d->splitk_exchange > 2 || d->split_clusters < 0 ||
        d->split_clusters > 2)
        return MLP_ERR_INVALID_ARG;
    // k-slices on separate clusters: the queue protocol on CTA pairs over one 256-row panel
    if (d->split_clusters == 2 && (d->mode != MLP_MODE_PIPELINED || d->cta_pair == 1 || !pair_ok || d->M > 2 * bm))
        return MLP_ERR_UNSUPPORTED;

    mlp_chain *h = new (std::nothrow) mlp_chain();
    if (!h)
        return MLP_ERR_OOM;
    h->desc = *d;
    h->S = S;
    h->fault_armed = (d->debug_flags & MLP_DEBUG_DROP_DECREMENT) != 0;
    h->device = d->device;
    if (cudaSetDevice(h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        release(h);
        return MLP_ERR_CUDA;
    }
    int cc_major = 0, cc_minor = 0, smem_optin = 0;
    cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, h->device);
    cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, h->device);
    cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
    if (cc_major != 10 || cc_minor != 3) {  // the binary is built for sm_103a only
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }

    h->bm = bm;
    h->tiles_m = static_cast<int>((d->M + bm - 1) / bm);   // single-CTA tiles; pairs are decided below
    // The device maximum, so that handles with different ring depths can share the kernel.
    if (cudaFuncSetAttribute(mlpc::chain_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mlpc::chain_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) !=
            cudaSuccess) {
        release(h);
        return MLP_ERR_CUDA;
    }
    // Co-resident clusters of 1, 2, 4, 8 CTAs (one CTA per SM; a cluster stays within a GPC).
    int clusters[4] = {h->num_sms, 0, 0, 0};
    for (int li = 1; li < 4; ++li) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1u << li;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((1u << li) * 8, 1, 1);
        cfg.blockDim = dim3(mlpc::kThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem_optin);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters[li], mlpc::chain_kernel<1>, &cfg) != cudaSuccess)
            clusters[li] = 0;
    }
    cudaGetLastError();
    // The same for CTA-pair clusters of 2, 4 and 8 CTAs (pair x k-slices).
    int clusters2[4] = {0, 0, 0, 0};
    if (pair_ok) {
        for (int li = 1; li < 4; ++li) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1u << li;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3((1u << li) * 8, 1, 1);
            cfg.blockDim = dim3(mlpc::kThreads, 1, 1);
            cfg.dynamicSmemBytes = static_cast<size_t>(smem_optin);
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&clusters2[li], mlpc::chain_kernel<2>, &cfg) != cudaSuccess)
                clusters2[li] = 0;
        }
        cudaGetLastError();
    }
    // Two plans, each stage's tile width and split from the cost model: one CTA per tile, and CTA
    // pairs.  Pairs run where asked for, or by default where the model, with the ring depth each
    // plan leaves, puts them at least 3 % ahead: prefill and the GeLU chain (a third less fill per
    // k block) and the Llama MLP with its down-projection's four k-slices on separate clusters
    // (in one cluster they would need clusters of 8, and only 15 of those fit: 120 CTAs), not
    // decode (a 256-row pair tile over 128 rows).
    int bn1[mlpc::kMaxStages] = {}, sp1[mlpc::kMaxStages] = {}, bn2[mlpc::kMaxStages] = {}, sp2[mlpc::kMaxStages] = {};
    int bn2x[mlpc::kMaxStages] = {}, sp2x[mlpc::kMaxStages] = {};
    double t1 = 0.0, t2 = pair_ok ? 0.0 : 1e30;
    const int64_t tiles_m1 = h->tiles_m, tiles_m2 = (d->M + 2 * bm - 1) / (2 * bm);
    // A third plan for pairs: k-slices on separate clusters of two (each a cluster item of its
    // own), which lifts the cluster-size limit on split pair tiles.  Only where a cluster can hold
    // no more than one item of such a stage (see StageParams::xsplit): the queue protocol, one
    // 256-row panel (every boundary one scoreboard group), a one-wave split stage.
    const bool xs_ok = pair_ok && d->mode == MLP_MODE_PIPELINED && tiles_m2 == 1 && d->split_clusters != 1;
    if (d->split_clusters == 2 && (!xs_ok || d->cta_pair == 1)) {
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }
    int clusters2x[4] = {0, 0, 0, 0};   // pair x S CTAs per tile, all resident as clusters of two
    double t2x = xs_ok ? 0.0 : 1e30;
    for (int s = 0; s < S; ++s) {
        const int tn = d->tile_n[s], ks = d->k_split[s];
        // tile widths: multiples of 32 up to 256 (a gated GEMM: 32, 64 or 128, its gate and up tiles
        // lying back to back as one tile twice as wide)
        const bool tn_ok = tn == 0 || (tn % 32 == 0 && tn <= 256 &&
                                       (!(d->gated && s == 0) || tn == 32 || tn == 64 || tn == 128));
        if (!tn_ok || (ks != 0 && ks != 1 && ks != 2 && ks != 4 && ks != 8)) {
            release(h);
            return !tn_ok ? MLP_ERR_UNSUPPORTED : MLP_ERR_INVALID_ARG;
        }
        // a gated GEMM issues two MMAs per k step into two accumulators: unsplit, at most 128 wide
        const bool gate_s = d->gated && s == 0;
        const int tn_s = gate_s && tn == 0 ? 128 : tn;
        const int ks_s = gate_s ? 1 : ks;
        t1 += choose_tiles(tiles_m1, bm, d->dims[s], d->dims[s + 1], clusters, tn_s, ks_s, &bn1[s], &sp1[s]);
        // a gated GEMM on pairs is costed as a plain pair GEMM twice as wide over the gate and up
        // columns side by side (the MMA's width), unsplit, and its tile is half that width
        const int64_t n2 = gate_s ? 2 * d->dims[s + 1] : d->dims[s + 1];
        const int tn2 = gate_s ? 2 * (tn ? tn : 128) : tn, ks2 = gate_s ? 1 : ks;
        if (t2 < 1e29) {
            t2 += choose_tiles(tiles_m2, bm, d->dims[s], n2, clusters2, tn2, ks2, &bn2[s], &sp2[s], 2, 0, 0.33);
            if (gate_s)
                bn2[s] /= 2;
        }
        if (t2x < 1e29) {
            for (int li = 1; li < 4; ++li)
                clusters2x[li] = clusters2[1] >> (li - 1);
            t2x += choose_tiles(tiles_m2, bm, d->dims[s], n2, clusters2x, tn2, ks2, &bn2x[s], &sp2x[s], 2, 0, 0.33, true);
            if (gate_s)
                bn2x[s] /= 2;
        }
    }
    // slices on separate clusters where asked for, or where that plan is better than the other
    // pair plan (it can only differ where a stage splits)
    bool use_x = false;
    if (t2x < 1e29) {
        bool splits = false;
        for (int s = 0; s < S; ++s)
            splits = splits || sp2x[s] > 1;
        use_x = d->split_clusters == 2 ? true : (splits && t2x < 0.999 * t2);
    }
    if (d->split_clusters == 2 && t2x >= 1e29) {
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }
    if (use_x) {
        for (int s = 0; s < S; ++s) {
            bn2[s] = bn2x[s];
            sp2[s] = sp2x[s];
        }
        t2 = t2x;
        for (int li = 1; li < 4; ++li)
            clusters2[li] = clusters2x[li];
    }
    bool pair_auto = false;
    if (d->cta_pair == 0 && pair_auto_ok && t1 < 1e29 && t2 < 1e29) {
        const size_t ring_bytes = static_cast<size_t>(smem_optin) - 1024 - 4 * mlpc::kEpiStageBytes - sizeof(mlpc::Ctrl);
        int mb1 = 0, mb2 = 0;   // widest B tile of a ring slot (a gated GEMM's: gate and up)
        for (int s = 0; s < S; ++s) {
            const int g = d->gated && s == 0 ? 2 : 1;
            mb1 = std::max(mb1, g * bn1[s]);
            mb2 = std::max(mb2, g * bn2[s]);
        }
        const int slots1 = static_cast<int>(std::min<size_t>(mlpc::kMaxPipe, ring_bytes / (bm * 128 + 128 * mb1)));
        const int slots2 = static_cast<int>(std::min<size_t>(mlpc::kMaxPipe, ring_bytes / (bm * 128 + 64 * mb2)));
        double e1 = 0.0, e2 = 0.0;
        for (int s = 0; s < S; ++s) {
            int b, k;
            const int g = d->gated && s == 0 ? 2 : 1;
            e1 += choose_tiles(tiles_m1, bm, d->dims[s], d->dims[s + 1], clusters, bn1[s], sp1[s], &b, &k, 1, slots1);
            e2 += choose_tiles(tiles_m2, bm, d->dims[s], g * d->dims[s + 1], clusters2, g * bn2[s], sp2[s], &b, &k, 2,
                               slots2, 0.33, use_x);
        }
        pair_auto = e2 < 0.97 * e1;
    }
    const int pair = (d->cta_pair == 2 || pair_auto || (use_x && d->split_clusters == 2)) ? 2 : 1;
    if ((pair == 2 ? t2 : t1) >= 1e29) {
        release(h);
        return MLP_ERR_UNSUPPORTED;   // no valid tile / split for this request
    }
    const int tile_rows = pair * bm;
    h->pair = pair;
    h->tiles_m = static_cast<int>((d->M + tile_rows - 1) / tile_rows);
    for (int s = 0; s < S; ++s) {
        const int bn = pair == 2 ? bn2[s] : bn1[s], split = pair == 2 ? sp2[s] : sp1[s];
        h->BN[s] = bn;
        h->b_swz[s] = bn >= 64 ? 128 : 64;
        h->tiles_n[s] = static_cast<int>((d->dims[s + 1] + bn - 1) / bn);
        h->k_blocks[s] = static_cast<int>((d->dims[s] + mlpc::kBK - 1) / mlpc::kBK);
        h->max_bn = std::max(h->max_bn, bn);
        h->split[s] = split;
        h->kb_per_split[s] = (h->k_blocks[s] + split - 1) / split;
        h->xsplit[s] = pair == 2 && use_x && split > 1;
        h->cs = std::max(h->cs, pair * (h->xsplit[s] ? 1 : split));
    }
    if (pair == 2)
        for (int li = 1; li < 4; ++li)
            clusters[li] = clusters2[li];
    for (int s = 0; s < S; ++s) {
        const int tiles = h->tiles_m * h->tiles_n[s];
        if (h->xsplit[s]) {   // a cluster item is one slice of one tile
            h->items[s] = tiles * h->split[s];
            continue;
        }
        const int tpi = h->cs / (pair * h->split[s]);
        h->items[s] = (tiles + tpi - 1) / tpi;
    }
    const uint32_t a_bytes = static_cast<uint32_t>(bm * mlpc::kBK * 2);
    // a pair's CTA loads half of B; a width that is not a multiple of the 64-column weight box
    // loads its last box whole
    auto padded_cols = [](int bn) { return bn >= 64 ? (bn + 63) / 64 * 64 : bn; };
    const int b_cols = padded_cols(h->max_bn / pair);
    h->stage_bytes = a_bytes + static_cast<uint32_t>(mlpc::kBK * b_cols * 2);
    // Two k blocks per fill where asked for (tile_k = 128) and the GEMM allows it: one CTA per tile,
    // a plain stage, K a multiple of 128 with every k-slice an even number of blocks, and a B tile
    // of whole weight boxes (the copy views need them).
    for (int s = 0; s < S; ++s) {
        const int box_cols = h->b_swz[s] / 2;
        const bool boxes = d->weight_layout == 1 || (d->dims[s + 1] % box_cols == 0 && h->BN[s] % box_cols == 0);
        const bool ok = pair == 1 && deep_ok && !(d->gated && s == 0) && d->dims[s] % 128 == 0 &&
                        h->kb_per_split[s] % 2 == 0 && boxes;
        h->kpf[s] = d->tile_k == 128 && ok ? 2 : 1;
        if (h->kpf[s] == 2)
            h->stage_bytes = std::max(h->stage_bytes, 2u * (a_bytes + static_cast<uint32_t>(mlpc::kBK * padded_cols(h->BN[s]) * 2)));
    }
    if (d->gated)   // the gated stage's ring slot holds gate and up weight tiles (a pair's CTA: one of them)
        h->stage_bytes = std::max(h->stage_bytes, a_bytes + static_cast<uint32_t>((pair == 2 ? 1 : 2) * mlpc::kBK * h->BN[0] * 2));
    h->n_w = S + (d->gated ? 1 : 0);
    // Split tiles reduce through global memory unless the shared-memory exchange is asked for.
    // (Distributed shared memory stores measured slower on the decode workload, 43.9 against
    // 40.2 us with the same ring depth: a warp's st.shared::cluster of 512 bytes costs more than
    // its global store, and the 64 KB receive buffer takes two ring slots.)
    if (d->splitk_exchange == 2)
        for (int s = 0; s < S; ++s)
            if (h->split[s] > 1) {
                if (static_cast<uint32_t>(h->BN[s] * bm * 4) > mlpc::kRecvBytes) {
                    release(h);
                    return MLP_ERR_UNSUPPORTED;
                }
                h->recv_bytes = mlpc::kRecvBytes;
            }
    const size_t fixed = 1024 + 4 * mlpc::kEpiStageBytes + h->recv_bytes + sizeof(mlpc::Ctrl);
    h->num_pipe = static_cast<int>(std::min<size_t>(mlpc::kMaxPipe, (smem_optin - fixed) / h->stage_bytes));
    if (d->pipe_stages)
        h->num_pipe = std::min(h->num_pipe, d->pipe_stages);
    h->acc_split = d->acc_split == 2 ? 2 : 1;
    h->acc_cols = std::max(h->acc_split * h->max_bn, d->gated ? 2 * h->BN[0] : 0);
    if (h->acc_cols & (h->acc_cols - 1))   // the second accumulator starts on a power-of-two column, as for the other widths
        h->acc_cols = (h->acc_cols + 127) / 128 * 128;
    if (2 * h->acc_cols > 512) {
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }
    if (h->num_pipe < 2) {
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }
    h->smem = mlpc::chain_smem_bytes(h->num_pipe, h->stage_bytes, h->recv_bytes);

    h->tmem_cols = 32;
    while (h->tmem_cols < static_cast<uint32_t>(2 * h->acc_cols))
        h->tmem_cols *= 2;
    h->stage_base[0] = 0;
    h->tile_base[0] = 0;
    for (int s = 0; s < S; ++s) {
        h->stage_base[s + 1] = h->stage_base[s] + h->items[s];
        h->tile_base[s + 1] = h->tile_base[s] + h->tiles_m * h->tiles_n[s];
    }
    const int total = h->tile_base[S];
    const int total_items = h->stage_base[S];
    h->max_clusters = clusters[h->cs == 1 ? 0 : h->cs == 2 ? 1 : h->cs == 4 ? 2 : 3];
    if (h->max_clusters < 1) {
        release(h);
        return MLP_ERR_UNSUPPORTED;
    }
    if (d->grid_ctas) {
        if (d->grid_ctas % h->cs) {
            release(h);
            return MLP_ERR_INVALID_ARG;
        }
        h->grid = d->grid_ctas;
    } else {
        h->grid = std::min(h->max_clusters, total_items) * h->cs;
    }
    if (is_pipelined(d->mode) && h->grid / h->cs > h->max_clusters) {
        release(h);  // the pipelined grid must be co-resident
        return MLP_ERR_INVALID_ARG;
    }
    for (int s = 0; s < S; ++s)
        if (h->xsplit[s] && h->items[s] > h->grid / h->cs) {
            release(h);  // slices on separate clusters need a cluster for every item of their stage
            return MLP_ERR_UNSUPPORTED;
        }
    h->raster_group = d->raster_group ? d->raster_group : default_raster_group(h->tiles_m, h->items[0], h->grid / h->cs);

    // dependency arrays (host), then one device block for all library-owned state
    size_t bytes = 8 * sizeof(uint32_t);
    for (int b = 0; b + 1 < S; ++b) {
        const int64_t nnz = mlp_deps_build(d->M, d->dims[b + 1], d->dims[b + 2], tile_rows, h->BN[b], tile_rows,
                                           h->BN[b + 1], nullptr, nullptr, 0, nullptr);
        if (nnz < 0) {
            release(h);
            return MLP_ERR_INVALID_ARG;
        }
        h->off[b].resize(static_cast<size_t>(h->tiles_m) * h->tiles_n[b] + 1);
        h->tgt[b].resize(static_cast<size_t>(std::max<int64_t>(nnz, 1)));
        h->init[b].resize(static_cast<size_t>(h->tiles_m) * h->tiles_n[b + 1]);
        mlp_deps_build(d->M, d->dims[b + 1], d->dims[b + 2], tile_rows, h->BN[b], tile_rows, h->BN[b + 1],
                       h->off[b].data(), h->tgt[b].data(), nnz, h->init[b].data());
        h->tgt[b].resize(static_cast<size_t>(nnz));
        // The first stage's raster walks groups of rg row panels column by column, so those
        // panels' consumers become ready together: one scoreboard group per rg panels, pushed
        // column by column so that neighbouring queue slots share a weight slab in L2.
        const int rg = h->raster_group;
        h->grp[b] = mlpc::scoreboard_groups(h->off[b].data(), h->tgt[b].data(), static_cast<int32_t>(h->off[b].size() - 1),
                                            static_cast<int32_t>(h->init[b].size()), h->tiles_n[b + 1], rg);
        const mlpc::DepGroups &G = h->grp[b];
        bytes = align_up(bytes, 256) + G.pg_off.size() * 4;
        bytes = align_up(bytes, 256) + std::max<size_t>(G.pg_tgt.size(), 1) * 4;
        bytes = align_up(bytes, 256) + G.grp_off.size() * 4;
        bytes = align_up(bytes, 256) + G.grp_mem.size() * 4;
        bytes = align_up(bytes, 256) + G.grp_init.size() * 4;      // init
        bytes = align_up(bytes, 256) + G.grp_init.size() * 4;      // count
        bytes = align_up(bytes, 256) + G.cons_grp.size() * 4;      // consumer -> group
        bytes = align_up(bytes, 256) + h->init[b].size() * 8;      // queue
        bytes = align_up(bytes, 256) + 4;                          // tail
        bytes = align_up(bytes, 256) + (h->off[b].size() - 1) * 4; // ready (K-granular mode)
    }
    for (int s = 0; s < S; ++s)   // slices on separate clusters: release counters per tile and half
        if (h->xsplit[s])
            bytes = align_up(bytes, 256) + static_cast<size_t>(h->tiles_m) * h->tiles_n[s] * pair * 4;
    if (d->debug_flags & MLP_DEBUG_EVENT_LOG) {
        h->n_events = static_cast<size_t>(total) + static_cast<size_t>(h->grid);   // tiles, then CTAs
        bytes = align_up(bytes, 256) + h->n_events * sizeof(mlpc::EventRec);
    }
    // split-K partial sums: per stage that splits, one 128 x max_bn fp32 buffer per CTA slot, or
    // with slices on separate clusters one per slice of every tile (written once per run)
    const int cta_slots = std::max(h->grid, h->max_clusters * h->cs);
    auto partial_bytes = [&](int s) {
        const size_t bufs = h->xsplit[s] ? static_cast<size_t>(h->tiles_m) * h->tiles_n[s] * h->split[s] * pair
                                         : static_cast<size_t>(cta_slots);
        return bufs * bm * h->max_bn * sizeof(float);
    };
    auto global_partials = [&](int s) {
        return h->split[s] > 1 && !(h->recv_bytes && static_cast<uint32_t>(h->BN[s] * bm * 4) <= h->recv_bytes);
    };
    for (int s = 0; s < S; ++s)
        if (global_partials(s))
            bytes = align_up(bytes, 256) + partial_bytes(s);
    if (cudaMalloc(&h->dev_block, bytes) != cudaSuccess) {
        h->dev_block = nullptr;
        release(h);
        return MLP_ERR_OOM;
    }
    uint8_t *p = static_cast<uint8_t *>(h->dev_block);
    size_t o = 0;
    h->d_ctrl = reinterpret_cast<uint32_t *>(p);
    o = 8 * sizeof(uint32_t);
    bool ok = true;
    for (int b = 0; b + 1 < S; ++b) {
        auto take = [&](size_t n) {
            o = align_up(o, 256);
            void *r = p + o;
            o += n;
            return r;
        };
        const mlpc::DepGroups &G = h->grp[b];
        DeviceBoundary &db = h->db[b];
        db.groups = G.grp_init.size();
        db.consumers = h->init[b].size();
        db.pg_off = static_cast<int32_t *>(take(G.pg_off.size() * 4));
        db.pg_tgt = static_cast<int32_t *>(take(std::max<size_t>(G.pg_tgt.size(), 1) * 4));
        db.grp_off = static_cast<int32_t *>(take(G.grp_off.size() * 4));
        db.grp_mem = static_cast<int32_t *>(take(G.grp_mem.size() * 4));
        db.grp_init = static_cast<int32_t *>(take(G.grp_init.size() * 4));
        db.count = static_cast<uint32_t *>(take(G.grp_init.size() * 4));
        db.cgrp = static_cast<int32_t *>(take(G.cons_grp.size() * 4));
        db.queue = static_cast<unsigned long long *>(take(db.consumers * 8));
        db.tail = static_cast<uint32_t *>(take(4));
        db.producers = h->off[b].size() - 1;
        db.ready = static_cast<uint32_t *>(take(db.producers * 4));
        auto up = [&](int32_t *dst, const std::vector<int32_t> &v) {
            if (!v.empty())
                ok = ok && cudaMemcpy(dst, v.data(), v.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess;
        };
        up(db.pg_off, G.pg_off);
        up(db.pg_tgt, G.pg_tgt);
        up(db.grp_off, G.grp_off);
        up(db.grp_mem, G.grp_mem);
        up(db.cgrp, G.cons_grp);
        // A producer tile is released by each epilogue warp of each of its CTAs (every split-K
        // slice, both CTAs of a pair).
        std::vector<int32_t> releases(G.grp_init);
        for (int32_t &v : releases)
            v *= releases_per_tile(h, b);
        up(db.grp_init, releases);
    }
    for (int s = 0; s < S; ++s)
        if (h->xsplit[s]) {
            o = align_up(o, 256);
            h->xcount[s] = reinterpret_cast<uint32_t *>(p + o);
            o += static_cast<size_t>(h->tiles_m) * h->tiles_n[s] * pair * 4;
        }
    h->meta_bytes = o;
    if (h->n_events) {
        o = align_up(o, 256);
        h->d_events = reinterpret_cast<mlpc::EventRec *>(p + o);
        ok = ok && cudaMemset(h->d_events, 0, h->n_events * sizeof(mlpc::EventRec)) == cudaSuccess;
        o += h->n_events * sizeof(mlpc::EventRec);
    }
    for (int s = 0; s < S; ++s)
        if (global_partials(s)) {
            o = align_up(o, 256);
            h->partials[s] = reinterpret_cast<float *>(p + o);
            o += partial_bytes(s);
        }
    if (!ok || full_reset(h) != MLP_OK) {
        release(h);
        return MLP_ERR_CUDA;
    }
    if (d->mode == MLP_MODE_MICROBATCH) {
        const int rows_tiles = d->microbatch_rows / tile_rows;   // chunk rows in (pair) tiles
        h->chunk_tiles = rows_tiles;
        h->n_chunks = (h->tiles_m + rows_tiles - 1) / rows_tiles;
        h->events.assign(static_cast<size_t>(h->n_chunks) * S, nullptr);
        for (auto &e : h->events)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                ok = false;
        if (cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) != cudaSuccess)
            ok = false;
        for (int s = 1; s < S; ++s)
            if (cudaStreamCreateWithFlags(&h->side[s], cudaStreamNonBlocking) != cudaSuccess)
                ok = false;
        if (!ok) {
            release(h);
            return MLP_ERR_CUDA;
        }
    }
    *out = h;
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_workspace_size(mlp_chain_t h, size_t *bytes)
{
    if (!h || !bytes)
        return MLP_ERR_INVALID_ARG;
    size_t b = 0;
    for (int s = 1; s < h->S; ++s)
        b = align_up(b, 256) + static_cast<size_t>(h->desc.M) * h->desc.dims[s] * 2;
    *bytes = b;
    return MLP_OK;
}

// Consumers of boundary b skip the work-queue (queue protocol only): one scoreboard group, whose
// queue would list its members in a fixed order anyway, or no more consumer items than
// co-resident clusters, where every consumer item gets a cluster of its own and readiness order
// cannot give any cluster a better tile.
static bool queue_free(const mlp_chain *h, int b)
{
    if (h->desc.mode != MLP_MODE_PIPELINED)
        return false;
    return h->grp[b].grp_init.size() == 1 || h->items[b + 1] <= h->grid / h->cs;
}

static mlp_status prepare_params(mlp_chain *h, const void *X, const void *const *W, void *Y, void *ws)
{
    bool same = h->params_valid && X == h->c_X && Y == h->c_Y && ws == h->c_ws;
    for (int s = 0; s < h->n_w && same; ++s)
        same = W[s] == h->c_W[s];
    if (same)
        return MLP_OK;
    ChainParams &P = h->params;
    std::memset(&P, 0, sizeof(P));
    const mlp_chain_desc &d = h->desc;
    size_t wo = 0;
    const void *a_ptr = X;
    for (int s = 0; s < h->S; ++s) {
        void *out_ptr;
        if (s + 1 < h->S) {
            wo = align_up(wo, 256);
            out_ptr = static_cast<uint8_t *>(ws) + wo;
            wo += static_cast<size_t>(d.M) * d.dims[s + 1] * 2;
        } else {
            out_ptr = Y;
        }
        const bool deep = h->kpf[s] == 2;
        if (!(deep ? encode_rows_kblocks(&P.mapA[s], a_ptr, d.M, d.dims[s], h->bm)
                   : encode_2d(&P.mapA[s], a_ptr, d.M, d.dims[s], h->bm, mlpc::kBK, CU_TENSOR_MAP_SWIZZLE_128B)))
            return MLP_ERR_CUDA;
        int32_t b_3d = 0, u_3d = 0;
        auto encode_w = [&](CUtensorMap *m, const void *w, int32_t *is_3d) {
            *is_3d = 0;
            const int bn_cta = d.gated && s == 0 ? h->BN[s] : h->BN[s] / h->pair;   // the columns one CTA loads
            if (deep)
                return d.weight_layout == 1 ? encode_rows_kblocks(m, w, d.dims[s + 1], d.dims[s], bn_cta)
                                            : encode_w_kn_kblocks(m, w, d.dims[s], d.dims[s + 1], h->b_swz[s], bn_cta);
            return d.weight_layout == 1
                       ? encode_2d(m, w, d.dims[s + 1], d.dims[s], bn_cta, mlpc::kBK, CU_TENSOR_MAP_SWIZZLE_128B)
                       : encode_w_kn(m, w, d.dims[s], d.dims[s + 1], mlpc::kBK, h->b_swz[s], bn_cta, is_3d);
        };
        const bool gate_s = d.gated && s == 0;
        if (!encode_w(&P.mapB[s], W[s == 0 ? 0 : s + (d.gated ? 1 : 0)], &b_3d) ||
            (gate_s && !encode_w(&P.mapU, W[1], &u_3d)))
            return MLP_ERR_CUDA;
        mlpc::StageParams &sp = P.st[s];
        sp.b_3d = b_3d && (!gate_s || u_3d);   // gate and up maps share the stage's copy shape
        if (gate_s && b_3d != u_3d &&
            !(encode_2d(&P.mapB[s], W[0], d.dims[s], d.dims[s + 1], mlpc::kBK, h->b_swz[s] / 2,
                        h->b_swz[s] == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B) &&
              encode_2d(&P.mapU, W[1], d.dims[s], d.dims[s + 1], mlpc::kBK, h->b_swz[s] / 2,
                        h->b_swz[s] == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)))
            return MLP_ERR_CUDA;
        sp.M = static_cast<int32_t>(d.M);
        sp.K = static_cast<int32_t>(d.dims[s]);
        sp.N = static_cast<int32_t>(d.dims[s + 1]);
        sp.BN = h->BN[s];
        sp.tiles_m = h->tiles_m;
        sp.tiles_n = h->tiles_n[s];
        sp.k_blocks = h->k_blocks[s];
        sp.b_swz = h->b_swz[s];
        sp.b_kmajor = d.weight_layout == 1;
        // the CTAs of one tile: its k-slices, each a pair with CTA pairs (rank 2 q + h: slice q, half h)
        sp.split = h->pair * h->split[s];
        sp.kb_per_split = h->kb_per_split[s];
        sp.tiles_per_item = h->xsplit[s] ? 1 : h->cs / (h->pair * h->split[s]);
        sp.items = h->items[s];
        sp.xsplit = h->xsplit[s] ? 1 : 0;
        sp.xcount = h->xcount[s];
        sp.partials = h->partials[s];
        sp.dsmem_reduce = h->split[s] > 1 && h->recv_bytes && static_cast<uint32_t>(h->BN[s] * h->bm * 4) <= h->recv_bytes;
        sp.out = static_cast<__nv_bfloat16 *>(out_ptr);
        sp.gelu = d.epilogue == MLP_EPI_GELU_TANH && !gate_s;
        sp.gated = gate_s;
        sp.kpf = h->kpf[s];
        sp.residual = (d.residual && s + 1 == h->S) ? static_cast<const __nv_bfloat16 *>(X) : nullptr;
        a_ptr = out_ptr;
    }
    for (int b = 0; b + 1 < h->S; ++b) {
        P.bd[b].pg_off = h->db[b].pg_off;
        P.bd[b].pg_tgt = h->db[b].pg_tgt;
        P.bd[b].grp_off = h->db[b].grp_off;
        P.bd[b].grp_mem = h->db[b].grp_mem;
        P.bd[b].grp_init = h->db[b].grp_init;
        P.bd[b].count = h->db[b].count;
        P.bd[b].cgrp = h->db[b].cgrp;
        P.bd[b].queue = h->db[b].queue;
        P.bd[b].tail = h->db[b].tail;
        P.bd[b].slots_per_run = static_cast<uint32_t>(h->db[b].consumers);
        P.bd[b].ready = h->db[b].ready;
        P.bd[b].ready_quota = static_cast<uint32_t>(releases_per_tile(h, b));
        P.bd[b].queue_free = queue_free(h, b) ? 1 : 0;
    }
    P.num_stages = h->S;
    for (int s = 0; s <= h->S; ++s) {
        P.stage_base[s] = h->stage_base[s];
        P.tile_base[s] = h->tile_base[s];
    }
    P.cs = h->cs;
    P.partial_floats = h->bm * h->max_bn;
    P.bm = h->bm;
    P.pair = h->pair;
    P.a_bytes = static_cast<uint32_t>(h->bm * mlpc::kBK * 2);
    P.recv_bytes = h->recv_bytes;
    // Grouped first-stage raster: a weight column slab is reused from L2 by the panels of a group
    // instead of being streamed again per panel.
    P.raster_group = h->raster_group;
    P.num_pipe = h->num_pipe;
    P.stage_bytes = h->stage_bytes;
    P.tmem_cols = h->tmem_cols;
    P.acc_stride = h->acc_cols;
    P.acc_split = h->acc_split;
    P.sub_stride = h->max_bn;
    P.drop_tile = -1;
    P.timeout_ns = static_cast<uint64_t>(d.timeout_us ? d.timeout_us : 2000000u) * 1000ull;
    P.ticket = h->d_ctrl + 0;
    P.status = h->d_ctrl + 1;
    P.seq = h->d_ctrl + 2;
    P.launches = reinterpret_cast<unsigned long long *>(h->d_ctrl + 4);
    P.tickets_per_run = static_cast<uint32_t>(h->stage_base[h->S]);
    P.events = h->d_events;
    P.meta = reinterpret_cast<const uint8_t *>(h->d_ctrl);
    P.meta_bytes = static_cast<uint32_t>(h->meta_bytes);
    h->c_X = X;
    h->c_Y = Y;
    h->c_ws = ws;
    for (int s = 0; s < h->n_w; ++s)
        h->c_W[s] = W[s];
    h->params_valid = true;
    return MLP_OK;
}

static bool launch(const ChainParams &P, int grid, size_t smem, cudaStream_t st)
{
    if (P.cs == 1 && !P.pdl_wait) {
        mlpc::chain_kernel<1><<<grid, mlpc::kThreads, smem, st>>>(P);
        return cudaGetLastError() == cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (P.cs > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(P.cs);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (P.pdl_wait) {   // a programmatic dependent of the previous launch on this stream
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(mlpc::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, P.pair == 2 ? mlpc::chain_kernel<2> : mlpc::chain_kernel<1>, P) == cudaSuccess &&
           cudaGetLastError() == cudaSuccess;
}

// CTAs of a non-pipelined launch over `items` cluster items.
static int static_grid(const mlp_chain *h, int items)
{
    if (h->desc.grid_ctas)
        return h->desc.grid_ctas;
    return std::min(h->max_clusters, std::max(items, 1)) * h->cs;
}

extern "C" mlp_status mlp_chain_run(mlp_chain_t h, const void *X, const void *const *W, void *Y, void *workspace,
                                    void *stream)
{
    if (!h || !X || !W || !Y)
        return MLP_ERR_INVALID_ARG;
    if (h->S > 1 && !workspace)
        return MLP_ERR_INVALID_ARG;
    auto misaligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
    if (misaligned(X) || misaligned(Y) || (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return MLP_ERR_INVALID_ARG;
    for (int s = 0; s < h->n_w; ++s)
        if (!W[s] || misaligned(W[s]))
            return MLP_ERR_INVALID_ARG;
    if (cudaSetDevice(h->device) != cudaSuccess)
        return MLP_ERR_CUDA;
    const mlp_status ps = prepare_params(h, X, W, Y, workspace);
    if (ps != MLP_OK)
        return ps;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ChainParams P = h->params;
    P.pdl_wait = 0;
    P.pdl_trigger = 0;
    if (is_pipelined(h->desc.mode)) {
        P.pipelined = 1;
        P.kwait = h->desc.mode == MLP_MODE_PIPELINED_KWAIT;
        P.lamport = h->desc.mode == MLP_MODE_PIPELINED_LAMPORT;
        P.force_reload = P.lamport && (h->desc.debug_flags & MLP_DEBUG_FORCE_RELOAD) != 0;
        if (P.lamport && h->S > 1) {
            size_t bytes = 0;
            mlp_chain_workspace_size(h, &bytes);
            const size_t n16 = bytes / 16;   // every intermediate is a multiple of 16 bytes
            const int blocks = static_cast<int>(std::min<size_t>(4 * h->num_sms, (n16 + 255) / 256));
            fill_sentinel_kernel<<<std::max(blocks, 1), 256, 0, st>>>(static_cast<uint4 *>(workspace), n16);
            if (cudaGetLastError() != cudaSuccess)
                return MLP_ERR_CUDA;
        }
        if (h->fault_armed) {
            P.drop_tile = h->desc.drop_tile;
            h->fault_armed = false;
        }
        P.first_stage = 0;
        P.m_tile_begin = 0;
        P.m_tile_end = h->tiles_m;
        return launch(P, h->grid, h->smem, st) ? MLP_OK : MLP_ERR_CUDA;
    }
    P.pipelined = 0;
    if (h->desc.mode == MLP_MODE_SEQUENTIAL || h->desc.mode == MLP_MODE_SEQUENTIAL_PDL) {
        const bool pdl = h->desc.mode == MLP_MODE_SEQUENTIAL_PDL;
        for (int s = 0; s < h->S; ++s) {
            P.first_stage = s;
            P.m_tile_begin = 0;
            P.m_tile_end = h->tiles_m;
            P.pdl_wait = pdl && s > 0;
            P.pdl_trigger = pdl && s + 1 < h->S;
            if (!launch(P, static_grid(h, h->items[s]), h->smem, st))
                return MLP_ERR_CUDA;
        }
        return MLP_OK;
    }
    // micro-batch: stage s of chunk i runs on stream s after stage s-1 of chunk i
    if (cudaEventRecord(h->fork, st) != cudaSuccess)
        return MLP_ERR_CUDA;
    for (int s = 1; s < h->S; ++s)
        if (cudaStreamWaitEvent(h->side[s], h->fork, 0) != cudaSuccess)
            return MLP_ERR_CUDA;
    for (int i = 0; i < h->n_chunks; ++i) {
        P.m_tile_begin = i * h->chunk_tiles;
        P.m_tile_end = std::min(h->tiles_m, (i + 1) * h->chunk_tiles);
        for (int s = 0; s < h->S; ++s) {
            cudaStream_t ss = s == 0 ? st : h->side[s];
            if (s > 0 && cudaStreamWaitEvent(ss, h->events[static_cast<size_t>(i) * h->S + s - 1], 0) != cudaSuccess)
                return MLP_ERR_CUDA;
            P.first_stage = s;
            const int tiles = (P.m_tile_end - P.m_tile_begin) * h->tiles_n[s];
            const int tpi = h->cs / (h->pair * h->split[s]);
            if (!launch(P, static_grid(h, (tiles + tpi - 1) / tpi), h->smem, ss))
                return MLP_ERR_CUDA;
            if (cudaEventRecord(h->events[static_cast<size_t>(i) * h->S + s], ss) != cudaSuccess)
                return MLP_ERR_CUDA;
        }
    }
    // join: the last stage of the last chunk follows every other launch
    if (h->S > 1 &&
        cudaStreamWaitEvent(st, h->events[static_cast<size_t>(h->n_chunks - 1) * h->S + h->S - 1], 0) != cudaSuccess)
        return MLP_ERR_CUDA;
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_run_host(mlp_chain_t h, const void *X_host, const void *const *W, void *Y_host,
                                         void *X_dev, void *Y_dev, void *workspace, void *stream)
{
    if (!h || !X_host || !Y_host || !X_dev || !Y_dev)
        return MLP_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t xb = static_cast<size_t>(h->desc.M) * h->desc.dims[0] * 2;
    const size_t yb = static_cast<size_t>(h->desc.M) * h->desc.dims[h->S] * 2;
    if (cudaSetDevice(h->device) != cudaSuccess)
        return MLP_ERR_CUDA;
    // Page-locked host memory the device can address: the last GEMM's epilogue stores into it
    // directly, tile by tile as the tiles complete, so the transfer runs under the chain.
    void *y_direct = nullptr;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, Y_host) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
        attr.devicePointer && (reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u) == 0)
        y_direct = attr.devicePointer;
    cudaGetLastError();   // a pageable pointer is not an error here
    if (cudaMemcpyAsync(X_dev, X_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MLP_ERR_CUDA;
    const mlp_status r = mlp_chain_run(h, X_dev, W, y_direct ? y_direct : Y_dev, workspace, stream);
    if (r != MLP_OK || y_direct)
        return r;
    return cudaMemcpyAsync(Y_host, Y_dev, yb, cudaMemcpyDeviceToHost, st) == cudaSuccess ? MLP_OK : MLP_ERR_CUDA;
}

extern "C" mlp_status mlp_chain_check(mlp_chain_t h, void *stream)
{
    if (!h)
        return MLP_ERR_INVALID_ARG;
    if (cudaSetDevice(h->device) != cudaSuccess ||
        cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLP_ERR_CUDA;
    for (auto &s : h->side)
        if (s && cudaStreamSynchronize(s) != cudaSuccess)
            return MLP_ERR_CUDA;
    uint32_t status = 0;
    if (cudaMemcpy(&status, h->d_ctrl + 1, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLP_ERR_CUDA;
    if (status == 0)
        return MLP_OK;
    const mlp_status r = full_reset(h);
    if (r != MLP_OK)
        return r;
    return status == MLP_ERR_BAD_TILE ? MLP_ERR_BAD_TILE : MLP_ERR_TIMEOUT;
}

extern "C" mlp_status mlp_chain_get_deps(mlp_chain_t h, int32_t b, const int32_t **off, const int32_t **tgt,
                                         const int32_t **init, int32_t *P, int32_t *C)
{
    if (!h || b < 0 || b + 1 >= h->S)
        return MLP_ERR_INVALID_ARG;
    if (off)
        *off = h->off[b].data();
    if (tgt)
        *tgt = h->tgt[b].data();
    if (init)
        *init = h->init[b].data();
    if (P)
        *P = static_cast<int32_t>(h->off[b].size() - 1);
    if (C)
        *C = static_cast<int32_t>(h->init[b].size());
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_get_scoreboard(mlp_chain_t h, int32_t b, mlp_scoreboard *sb)
{
    if (!h || !sb || b < 0 || b + 1 >= h->S)
        return MLP_ERR_INVALID_ARG;
    const DeviceBoundary &db = h->db[b];
    const mlpc::DepGroups &G = h->grp[b];
    sb->producers = static_cast<int32_t>(db.producers);
    sb->consumers = static_cast<int32_t>(db.consumers);
    sb->groups = static_cast<int32_t>(db.groups);
    sb->edges = static_cast<int32_t>(G.pg_tgt.size());
    sb->releases_per_producer = releases_per_tile(h, b);
    if (!sb->pg_off || !sb->pg_tgt || !sb->grp_off || !sb->grp_mem || !sb->grp_target || !sb->cons_grp)
        return MLP_OK;
    // the tables as the kernel reads them: copied back from the device block
    auto down = [](int32_t *dst, const int32_t *src, size_t n) {
        return n == 0 || cudaMemcpy(dst, src, n * 4, cudaMemcpyDeviceToHost) == cudaSuccess;
    };
    if (cudaSetDevice(h->device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        !down(sb->pg_off, db.pg_off, db.producers + 1) || !down(sb->pg_tgt, db.pg_tgt, G.pg_tgt.size()) ||
        !down(sb->grp_off, db.grp_off, db.groups + 1) || !down(sb->grp_mem, db.grp_mem, db.consumers) ||
        !down(sb->grp_target, db.grp_init, db.groups) || !down(sb->cons_grp, db.cgrp, db.consumers))
        return MLP_ERR_CUDA;
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_get_event_log(mlp_chain_t h, mlp_event *buf, size_t cap, size_t *n)
{
    if (!h || !buf || !n || !h->d_events)
        return MLP_ERR_INVALID_ARG;
    static_assert(sizeof(mlp_event) == sizeof(mlpc::EventRec), "event record layout");
    if (cudaSetDevice(h->device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return MLP_ERR_CUDA;
    const size_t k = std::min(cap, h->n_events);
    if (cudaMemcpy(buf, h->d_events, k * sizeof(mlp_event), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLP_ERR_CUDA;
    *n = k;
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_get_info(mlp_chain_t h, mlp_chain_info *info)
{
    if (!h || !info)
        return MLP_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    info->num_gemms = h->S;
    info->tile_m = h->bm * h->pair;
    info->cta_pair = h->pair;
    info->raster_group = h->raster_group;
    info->tile_k = mlpc::kBK;
    for (int b = 0; b + 1 < h->S; ++b)
        info->queue_free[b] = queue_free(h, b) ? 1 : 0;
    for (int s = 0; s < h->S; ++s)
        info->split_across[s] = h->xsplit[s] ? 1 : 0;
    for (int s = 0; s < h->S; ++s) {
        info->fill_k[s] = mlpc::kBK * h->kpf[s];
        info->tile_k = std::max(info->tile_k, info->fill_k[s]);
        info->tile_n[s] = h->BN[s];
        info->tiles_m[s] = h->tiles_m;
        info->tiles_n[s] = h->tiles_n[s];
    }
    info->grid_ctas = h->grid;
    info->num_sms = h->num_sms;
    info->pipe_stages = h->num_pipe;
    info->smem_bytes = static_cast<int32_t>(h->smem);
    info->tmem_cols = static_cast<int32_t>(h->tmem_cols);
    info->launches_per_run = is_pipelined(h->desc.mode) ? (h->desc.mode == MLP_MODE_PIPELINED_LAMPORT && h->S > 1 ? 2 : 1)
                             : (h->desc.mode == MLP_MODE_SEQUENTIAL || h->desc.mode == MLP_MODE_SEQUENTIAL_PDL) ? h->S
                                                                   : h->S * h->n_chunks;
    info->cluster_size = h->cs;
    for (int s = 0; s < h->S; ++s)
        info->k_split[s] = h->split[s];
    return MLP_OK;
}

extern "C" mlp_status mlp_chain_destroy(mlp_chain_t h)
{
    if (!h)
        return MLP_ERR_INVALID_ARG;
    cudaSetDevice(h->device);
    for (auto &s : h->side)
        if (s)
            cudaStreamSynchronize(s);
    release(h);
    return MLP_OK;
}

// ============================================================================================
// Allocation-free entry point.
//
// Some callers cannot allocate device memory at the point where they run the chain: code that
// runs inside a custom allocator or memory-pool callback, a runtime that reserves every byte of
// device memory up front and forbids further cudaMalloc, or an embedding that must not touch
// the CUDA caching allocator of the host framework.  mlp_chain_run_noalloc serves them: it runs
// the two-GEMM chain in pipelined mode with all of its scratch (the intermediate H, the
// dependency array, scoreboard, work-queue, tickets and status word) inside the file-scope
// array below, which every GPU that loads this library holds until the process exits.
// ============================================================================================
namespace {

__device__ __align__(256) static uint8_t g_noalloc_scratch[MLP_NOALLOC_SCRATCH_BYTES];

// SM count per device ordinal (a property of the device, not of a context: safe to keep).
int g_noalloc_sms[64] = {};
std::mutex g_noalloc_mutex;

struct NoallocLayout {
    size_t ctrl, pg_off, pg_tgt, grp_off, grp_mem, grp_init, count, cgrp, queue, tail, h, total;
};

// Groups are the row panels (tiles_m of them); every producer feeds exactly its own panel.
NoallocLayout noalloc_layout(int64_t M, int64_t N1, int P, int C, int G)
{
    NoallocLayout L{};
    size_t o = 0;
    L.ctrl = o;  o += 8 * sizeof(uint32_t);
    o = align_up(o, 256); L.pg_off = o;   o += static_cast<size_t>(P + 1) * 4;
    o = align_up(o, 256); L.pg_tgt = o;   o += static_cast<size_t>(P) * 4;
    o = align_up(o, 256); L.grp_off = o;  o += static_cast<size_t>(G + 1) * 4;
    o = align_up(o, 256); L.grp_mem = o;  o += static_cast<size_t>(C) * 4;
    o = align_up(o, 256); L.grp_init = o; o += static_cast<size_t>(G) * 4;
    o = align_up(o, 256); L.count = o; o += static_cast<size_t>(G) * 4;
    o = align_up(o, 256); L.cgrp = o;  o += static_cast<size_t>(C) * 4;
    o = align_up(o, 256); L.queue = o; o += static_cast<size_t>(C) * 8;
    o = align_up(o, 256); L.tail = o;  o += 4;
    o = align_up(o, 256); L.h = o;     o += static_cast<size_t>(M) * N1 * 2;
    L.total = o;
    return L;
}

// Writes the whole protocol state of one run into the scratch: control words cleared, the
// grouped dependency array of equal-height row tiles (producer tile (m, n) feeds row panel m;
// panel m holds consumer tiles m*Cn .. m*Cn+Cn-1 and waits for its Pn producer tiles),
// counters and the epoch cleared, queue slots emptied.  Nothing of a previous call survives.
__global__ void noalloc_setup_kernel(uint8_t *base, NoallocLayout L, int Pn, int Cn, int tiles_m)
{
    const int P = tiles_m * Pn, C = tiles_m * Cn, G = tiles_m;
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(base + L.ctrl);
    int32_t *pg_off = reinterpret_cast<int32_t *>(base + L.pg_off);
    int32_t *pg_tgt = reinterpret_cast<int32_t *>(base + L.pg_tgt);
    int32_t *grp_off = reinterpret_cast<int32_t *>(base + L.grp_off);
    int32_t *grp_mem = reinterpret_cast<int32_t *>(base + L.grp_mem);
    int32_t *grp_init = reinterpret_cast<int32_t *>(base + L.grp_init);
    uint32_t *count = reinterpret_cast<uint32_t *>(base + L.count);
    int32_t *cgrp = reinterpret_cast<int32_t *>(base + L.cgrp);
    unsigned long long *queue = reinterpret_cast<unsigned long long *>(base + L.queue);
    const int stride = gridDim.x * blockDim.x;
    const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = i0; i < 8; i += stride)
        ctrl[i] = 0;
    if (i0 == 0)
        *reinterpret_cast<uint32_t *>(base + L.tail) = 0;
    for (int i = i0; i <= P; i += stride) {
        pg_off[i] = i;
        if (i < P)
            pg_tgt[i] = i / Pn;
    }
    for (int g = i0; g <= G; g += stride) {
        grp_off[g] = g * Cn;
        if (g < G) {
            grp_init[g] = Pn * mlpc::kEpiWarps;   // each epilogue warp of a tile releases its rows
            count[g] = 0u;                        // the epoch word is cleared too: run 0's target
        }
    }
    for (int c = i0; c < C; c += stride) {
        grp_mem[c] = c;
        cgrp[c] = c / Cn;
        queue[c] = 0;
    }
}

}  // namespace

extern "C" mlp_status mlp_chain_run_noalloc(int64_t M, int64_t K, int64_t N1, int64_t N2, const void *X,
                                            const void *W1, const void *W2, void *Y, int32_t sync_check,
                                            void *stream)
{
    if (M < 1 || M > (int64_t)1 << 30 || !X || !W1 || !W2 || !Y)
        return MLP_ERR_INVALID_ARG;
    const int64_t dims[3] = {K, N1, N2};
    for (int64_t d : dims)
        if (d < 8 || d % 8 != 0 || d > (int64_t)1 << 24)
            return MLP_ERR_INVALID_ARG;
    auto misaligned = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0; };
    if (misaligned(X) || misaligned(W1) || misaligned(W2) || misaligned(Y))
        return MLP_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return MLP_ERR_CUDA;

    // Set-up on the current device, every call: the scratch array's device address and the
    // kernel's shared-memory limit belong to the current context (a cudaDeviceReset makes a new
    // one), so neither is cached; only the SM count is.  Once the module is loaded these calls
    // allocate nothing.
    int num_sms = 0, smem_optin = 0;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (g_noalloc_sms[dev] == 0) {
            int major = 0, minor = 0;
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            if (major != 10 || minor != 3)
                return MLP_ERR_UNSUPPORTED;
            if (cudaDeviceGetAttribute(&g_noalloc_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return MLP_ERR_CUDA;
        }
        num_sms = g_noalloc_sms[dev];
    }
    void *scratch_ptr = nullptr;
    if (cudaGetSymbolAddress(&scratch_ptr, g_noalloc_scratch) != cudaSuccess || !scratch_ptr ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncSetAttribute(mlpc::chain_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) != cudaSuccess)
        return MLP_ERR_CUDA;

    // Tiling: the same choices mlp_chain_create makes for this shape.
    const int tiles_m = static_cast<int>((M + mlpc::kBM - 1) / mlpc::kBM);
    const int no_clusters[4] = {num_sms, 0, 0, 0};   // this entry point runs without clusters
    int bn[2] = {256, 256}, unused = 1;
    choose_tiles(tiles_m, mlpc::kBM, K, N1, no_clusters, 0, 1, &bn[0], &unused);
    choose_tiles(tiles_m, mlpc::kBM, N1, N2, no_clusters, 0, 1, &bn[1], &unused);
    const int tn[2] = {static_cast<int>((N1 + bn[0] - 1) / bn[0]), static_cast<int>((N2 + bn[1] - 1) / bn[1])};
    const int P = tiles_m * tn[0], C = tiles_m * tn[1];
    const NoallocLayout L = noalloc_layout(M, N1, P, C, tiles_m);
    if (L.total > MLP_NOALLOC_SCRATCH_BYTES)
        return MLP_ERR_INVALID_ARG;   // this shape needs more scratch than the static array holds

    const int max_bn = std::max(bn[0], bn[1]);
    const uint32_t stage_bytes = mlpc::kABytes + static_cast<uint32_t>(mlpc::kBK * max_bn * 2);
    const int num_pipe = static_cast<int>(std::min<size_t>(
        mlpc::kMaxPipe, (smem_optin - 1024 - 4 * mlpc::kEpiStageBytes - sizeof(mlpc::Ctrl)) / stage_bytes));   // no split: no receive buffer
    if (num_pipe < 2)
        return MLP_ERR_UNSUPPORTED;
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(2 * max_bn))
        tmem_cols *= 2;

    uint8_t *base = static_cast<uint8_t *>(scratch_ptr);
    void *H = base + L.h;
    ChainParams P_;
    std::memset(&P_, 0, sizeof(P_));
    const void *a_ptr[2] = {X, H};
    const void *w_ptr[2] = {W1, W2};
    void *o_ptr[2] = {H, Y};
    for (int s = 0; s < 2; ++s) {
        const int b_swz = bn[s] >= 64 ? 128 : 64;
        int32_t b_3d = 0;
        if (!encode_2d(&P_.mapA[s], a_ptr[s], M, dims[s], mlpc::kBM, mlpc::kBK, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_w_kn(&P_.mapB[s], w_ptr[s], dims[s], dims[s + 1], mlpc::kBK, b_swz, bn[s], &b_3d))
            return MLP_ERR_CUDA;
        mlpc::StageParams &sp = P_.st[s];
        sp.b_3d = b_3d;
        sp.M = static_cast<int32_t>(M);
        sp.K = static_cast<int32_t>(dims[s]);
        sp.N = static_cast<int32_t>(dims[s + 1]);
        sp.BN = bn[s];
        sp.tiles_m = tiles_m;
        sp.tiles_n = tn[s];
        sp.k_blocks = static_cast<int32_t>((dims[s] + mlpc::kBK - 1) / mlpc::kBK);
        sp.b_swz = b_swz;
        sp.out = static_cast<__nv_bfloat16 *>(o_ptr[s]);
        sp.split = 1;
        sp.kb_per_split = sp.k_blocks;
        sp.tiles_per_item = 1;
        sp.items = tiles_m * tn[s];
    }
    P_.bd[0].pg_off = reinterpret_cast<const int32_t *>(base + L.pg_off);
    P_.bd[0].pg_tgt = reinterpret_cast<const int32_t *>(base + L.pg_tgt);
    P_.bd[0].grp_off = reinterpret_cast<const int32_t *>(base + L.grp_off);
    P_.bd[0].grp_mem = reinterpret_cast<const int32_t *>(base + L.grp_mem);
    P_.bd[0].grp_init = reinterpret_cast<const int32_t *>(base + L.grp_init);
    P_.bd[0].count = reinterpret_cast<uint32_t *>(base + L.count);
    P_.bd[0].cgrp = reinterpret_cast<const int32_t *>(base + L.cgrp);
    P_.bd[0].queue = reinterpret_cast<unsigned long long *>(base + L.queue);
    P_.bd[0].tail = reinterpret_cast<uint32_t *>(base + L.tail);
    P_.num_stages = 2;
    P_.pipelined = 1;
    P_.m_tile_end = tiles_m;
    P_.stage_base[0] = 0;
    P_.stage_base[1] = P;
    P_.stage_base[2] = P + C;
    P_.tile_base[0] = 0;
    P_.tile_base[1] = P;
    P_.tile_base[2] = P + C;
    P_.cs = 1;
    P_.partial_floats = mlpc::kBM * max_bn;
    P_.bm = mlpc::kBM;
    P_.pair = 1;
    P_.a_bytes = mlpc::kABytes;
    P_.num_pipe = num_pipe;
    P_.stage_bytes = stage_bytes;
    P_.tmem_cols = tmem_cols;
    P_.acc_stride = max_bn;
    P_.acc_split = 1;
    P_.sub_stride = max_bn;
    P_.drop_tile = -1;
    P_.timeout_ns = 2000000000ull;
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(base + L.ctrl);
    P_.ticket = ctrl + 0;
    P_.status = ctrl + 1;
    P_.seq = ctrl + 2;
    P_.launches = reinterpret_cast<unsigned long long *>(ctrl + 4);
    P_.tickets_per_run = static_cast<uint32_t>(P + C);
    P_.bd[0].slots_per_run = static_cast<uint32_t>(C);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long work = std::max(C, P + 1);
    const int setup_blocks = static_cast<int>(std::min<long long>(1024, (work + 255) / 256));
    noalloc_setup_kernel<<<setup_blocks, 256, 0, st>>>(base, L, tn[0], tn[1], tiles_m);
    if (cudaGetLastError() != cudaSuccess)
        return MLP_ERR_CUDA;
    const int grid = std::min(num_sms, P + C);
    if (!launch(P_, grid, mlpc::chain_smem_bytes(num_pipe, stage_bytes, 0), st))
        return MLP_ERR_CUDA;
    if (!sync_check)
        return MLP_OK;
    uint32_t status = 0;
    if (cudaMemcpyAsync(&status, ctrl + 1, sizeof(status), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return MLP_ERR_CUDA;
    if (status == 0)
        return MLP_OK;
    return status == MLP_ERR_BAD_TILE ? MLP_ERR_BAD_TILE : MLP_ERR_TIMEOUT;
}
