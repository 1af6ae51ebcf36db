/*
 * mlp_chain.h -- C ABI of the CTA-pipelined GEMM chain library (libmlp_chain.so).
 *
 * What it computes.  A chain of S dependent GEMMs on one GPU,
 *     A_0 = X,   A_{s+1} = epi_s( A_s * W_s ),   Y = A_S,
 * with bf16 operands, fp32 accumulation and every intermediate stored as bf16.  S = 2 is the
 * two-layer GEMM standing in for an MLP block, Y = (X*W1)*W2, the running example of
 * "CTA-Pipelining: A Latency-Oriented Spatial Scaling Method for Multi-GPU Systems"
 * (arXiv 2607.07862, section III: the first GEMM's output is consumed directly by the next
 * GEMM; bf16 in/out with an fp32 accumulator, Fig. 2 set-up).  S > 2 is the multi-layer GEMM
 * of section IV (Fig. 3-4).  epi_s is the identity, or GeLU(tanh) on the fp32 accumulator
 * (MLP_EPI_GELU_TANH), and with `residual` the last stage also adds X before rounding.
 *
 * How it schedules (MLP_MODE_PIPELINED).  CTA-pipelining (section III-A and Fig. 1): every
 * stage boundary owns a dependency array (built on the host from the static tile dataflow), a
 * scoreboard of per-consumer-tile counters initialised from it, and a work-queue.  A producer
 * tile stores its output, fences, and decrements the counter of every consumer tile that reads
 * it; the decrement that reaches zero pushes that consumer's tile id onto the queue.  Consumer
 * CTAs poll the queue in a short prologue, adopt the dequeued tile id in place of their own
 * and run the unchanged GEMM body.  (Here the counters count releases up to an epoch-scaled
 * target instead of down to zero, one counter per group of consumer tiles with the same
 * producers, and a consumer acquires its group counter before it reads the producers' output;
 * mlp_chain_get_scoreboard returns those counters' tables.)  All stages run in ONE persistent,
 * warp-specialised kernel on one GPU (one CTA per SM): the pages put one layer per GPU instead.
 * MLP_MODE_SEQUENTIAL launches the same tile engine once per GEMM, back to back on one stream
 * (the pages' "two consecutive GEMMs" baseline, section III-C).  MLP_MODE_MICROBATCH splits
 * X into row chunks and overlaps GEMM s of chunk i with GEMM s+1 of chunk i-1 on separate
 * streams (static micro-batching, section IV, Fig. 3).  MLP_MODE_PIPELINED_KWAIT is the same
 * persistent grid with a finer dependency: a consumer tile takes its place in raster order (no
 * work-queue) and, before loading k block kb of its input, waits only for the producer tiles
 * that wrote those 64 columns, each counted ready once all of its epilogue warps released their
 * rows (the tile-granular dependency of section III-A refined to the consumer's k loop; its
 * weight tiles are requested before the wait).  Every mode uses the same tiles in the same
 * order of k, so Y is bit-identical across modes.
 *
 * MLP_MODE_SEQUENTIAL_PDL is the pages' two-kernel form (one kernel per layer, the consumer
 * launched while the producer still runs) without its flag polling across kernels, which
 * nothing makes safe on one GPU (co-residency of two grids is not guaranteed): GEMM s+1 is a
 * programmatic dependent launch of GEMM s.  Every CTA of GEMM s allows its dependents at start;
 * GEMM s+1's CTAs then take SMs as GEMM s's CTAs retire, run their set-up (barriers, TMEM,
 * descriptor prefetch) and wait in the TMA warp, before the first load of GEMM s's output, for
 * GEMM s to complete (griddepcontrol.wait, a hardware dependency).  Same tiles and k order as
 * MLP_MODE_SEQUENTIAL, so Y is bit-identical to it.
 *
 * MLP_MODE_PIPELINED_LAMPORT is the paper's Lamport-synchronisation alternative (section V):
 * the same queue protocol with no fence on either side.  run() first fills the intermediates
 * with bf16 -0.0 (one extra launch); producers store +0.0 for an exact -0.0 and publish without
 * a release; a consumer scans each 64-deep A tile it loads from an intermediate in shared
 * memory and re-loads it until no -0.0 is left, before the tensor cores read it.  Y is
 * bit-identical to the other modes except where an intermediate is an exact -0.0, which this
 * mode stores as +0.0.  The plain data race it relies on (a load that sees either the sentinel
 * or the final value, never an older one) is outside the PTX memory model, as on the pages.
 *
 * Conventions for every entry point.
 *   - Matrices are dense, row-major, bf16, with 16-byte aligned base pointers; every
 *     dimension except M must be a multiple of 8 (one 16-byte TMA unit).
 *   - Device pointers are CUDA device addresses on the handle's device; host pointers are
 *     ordinary process memory (pinned memory makes the copies asynchronous).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - The caller owns X, W[], Y and the workspace.  The library owns its device state
 *     (scoreboards, queues, tickets, status word, event log), allocated in create and freed in
 *     destroy.
 *   - Errors are returned, never thrown or trapped.  Device-side failures (a bounded wait that
 *     ran out, a bad dequeued tile id) set a sticky status word that mlp_chain_check reports;
 *     until then further runs of that handle do nothing.
 *   - A handle is not thread-safe, and two runs of one handle must not overlap on the GPU
 *     (they share one scoreboard).  Different handles are independent.
 */
#ifndef MLP_CHAIN_H_
#define MLP_CHAIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLP_MAX_GEMMS 4

typedef enum {
    MLP_OK = 0,
    MLP_ERR_INVALID_ARG = 1,  /* a size, pointer, alignment or option is not acceptable      */
    MLP_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement (dtype, tile) */
    MLP_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                             */
    MLP_ERR_OOM = 4,          /* device allocation failed                                      */
    MLP_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (dependency never satisfied)    */
    MLP_ERR_DEVICE_STATE = 6, /* the handle's device state is inconsistent (reset pending)     */
    MLP_ERR_BAD_TILE = 7      /* a dequeued tile id was out of range                           */
} mlp_status;

typedef enum { MLP_DT_BF16 = 1, MLP_DT_F32 = 2 } mlp_dtype;

typedef enum {
    MLP_MODE_PIPELINED = 0,   /* one persistent grid, scoreboard + work-queue (CTA-pipelining) */
    MLP_MODE_SEQUENTIAL = 1,  /* one launch per GEMM, back to back                              */
    MLP_MODE_MICROBATCH = 2,  /* row chunks, GEMM s+1 of chunk i overlaps GEMM s of chunk i+1   */
    MLP_MODE_PIPELINED_KWAIT = 3, /* one persistent grid, per-k-block producer waits, no queue  */
    MLP_MODE_PIPELINED_LAMPORT = 4, /* the queue protocol without fences: sentinel-filled
                                      intermediates, consumers validate what they load         */
    MLP_MODE_SEQUENTIAL_PDL = 5 /* one launch per GEMM, each later one a programmatic dependent
                                   launch of the one before (no spin on another kernel's flags) */
} mlp_mode;

typedef enum { MLP_EPI_NONE = 0, MLP_EPI_GELU_TANH = 1 } mlp_epilogue;

/* debug_flags bits */
#define MLP_DEBUG_EVENT_LOG 1u          /* record one mlp_event per tile (pipelined mode)        */
#define MLP_DEBUG_DROP_DECREMENT 2u     /* fault injection, first pipelined run of the handle
                                           only: first-stage producer tile `drop_tile` skips its
                                           scoreboard decrements, so its consumers never become
                                           ready and their bounded wait must end the run with
                                           MLP_ERR_TIMEOUT                                       */
#define MLP_DEBUG_FORCE_RELOAD 4u       /* MLP_MODE_PIPELINED_LAMPORT test hook: treat every
                                           consumer A tile as unfinished once, so each is loaded
                                           twice (exercises the re-load path; same results)       */

typedef struct {
    int64_t M;                          /* rows of X (any value >= 1)                           */
    int32_t num_gemms;                  /* S, 1..MLP_MAX_GEMMS                                   */
    int64_t dims[MLP_MAX_GEMMS + 1];    /* K, N1, N2, ...: W_s is dims[s] x dims[s+1]            */
    mlp_dtype in_dtype, acc_dtype, h_dtype, out_dtype; /* must be BF16, F32, BF16, BF16         */
    int32_t tile_m;                     /* rows per tile: 0 (= 128), 128, or 64 (tcgen05 MMAs of
                                           M = 64: half the activation bytes per tile, twice the
                                           row panels; micro-batch chunks of 64 rows)           */
    int32_t tile_n[MLP_MAX_GEMMS];      /* per GEMM: 0 (library choice) or a multiple of 32 up to
                                           256 (a gated GEMM: 32, 64 or 128); a width that is not
                                           a multiple of 64 loads its last 64-column weight box
                                           whole, one copy per box; the library chooses among
                                           32, 64, 128 and 256                                   */
    int32_t tile_k;                     /* k depth of one shared-memory ring fill: 0 or 64, or 128
                                           (two 64-deep blocks per fill, one copy per operand and
                                           one barrier phase for twice the bytes; fewer, larger
                                           ring slots).  128 applies to the GEMMs with K a multiple
                                           of 128, k-slices of an even number of 64-deep blocks,
                                           whole weight boxes per tile and no gate; the others
                                           fill 64 deep (mlp_chain_info.fill_k).  With CTA pairs,
                                           split accumulators or the K-granular and Lamport modes:
                                           UNSUPPORTED                                           */
    mlp_epilogue epilogue;              /* applied after every GEMM                              */
    int32_t residual;                   /* nonzero: last stage adds X (needs dims[S] == dims[0]) */
    mlp_mode mode;
    int32_t microbatch_rows;            /* MICROBATCH: rows per chunk, a multiple of tile_m     */
    int32_t device;                     /* CUDA device ordinal                                  */
    uint32_t debug_flags;               /* MLP_DEBUG_* bits                                     */
    int32_t drop_tile;                  /* with MLP_DEBUG_DROP_DECREMENT                         */
    uint32_t timeout_us;                /* bounded device waits; 0 = 2 000 000 (2 s)             */
    int32_t grid_ctas;                  /* 0 = one CTA per SM                                    */
    int32_t raster_group;               /* first-stage raster: 1 = row panels in order; g > 1 =
                                           groups of g row panels, column-major inside a group;
                                           0 = library choice (8 from 16 panels, 4 from 8;
                                           below 8 all panels when the first stage takes more
                                           than one wave, else 1; see mlp_chain_info);
                                           pipelined consumers are grouped the same way         */
    int32_t pipe_stages;                /* shared-memory ring depth: 0 = as deep as fits         */
    int32_t weight_layout;              /* 0: W_s stored dims[s] x dims[s+1] row-major (K x N);
                                           1: stored transposed, dims[s+1] x dims[s] row-major
                                           (N x K, the layout of nn.Linear.weight)             */
    int32_t k_split[MLP_MAX_GEMMS];     /* per GEMM: k-slices sharing one tile along its reduction
                                           dimension (split-K inside a thread-block cluster; each
                                           slice one CTA, or one CTA pair): 0 = library choice,
                                           else 1, 2, 4 or 8 with tile_n / k_split >= 32; partial
                                           sums are added in a fixed order, so results stay
                                           deterministic                                         */
    int32_t acc_split;                  /* 0/1: one fp32 accumulator per tile; 2: 16-deep k steps
                                           alternate between two accumulators that the epilogue
                                           adds (even + odd), so consecutive MMAs do not depend on
                                           each other; needs 4 * tile_n <= 512                    */
    int32_t gated;                      /* nonzero: the first GEMM is a gated linear unit with a
                                           SiLU gate (the SwiGLU MLP block): run() takes
                                           S + 1 weights, W[0] = gate and W[1] = up (both
                                           dims[0] x dims[1]), and A_1 = SiLU(X W[0]) * (X W[1])
                                           from two fp32 accumulators, rounded once; W[s + 1] is
                                           the weight of GEMM s >= 1.  The gated GEMM runs
                                           unsplit with tile_n <= 128 and acc_split 1; epilogue
                                           (GeLU) applies to the later GEMMs only                 */
    int32_t cta_pair;                   /* 0: library choice (one CTA per tile, or CTA pairs where
                                           its cost model puts them ahead; never for micro-batch
                                           chunks); 1: one CTA per tile; 2: CTA pairs (tcgen05
                                           cta_group::2), each pair computing a 256-row tile, each
                                           CTA loading its 128 rows of the activations and half of
                                           the weight tile's columns (tiles 128 or 256 wide; of a
                                           gated GEMM's tile, 64 or 128 wide, the leader loads the
                                           gate tile and the peer the up tile), so a k block's fill
                                           per SM shrinks by a third and the ring gets deeper.
                                           With k_split S a tile takes S pairs in one cluster of
                                           2 S <= 8 CTAs, or S clusters of 2 (split_clusters).  No
                                           split accumulators, 64-row tiles, K-granular or Lamport
                                           modes, or shared-memory split-K exchange (else
                                           UNSUPPORTED); micro-batch chunks are multiples of 256
                                           rows                                                  */
    int32_t splitk_exchange;            /* how split-K siblings add their partial sums (k_split
                                           > 1), always in sibling order, so both give the same
                                           bits: 0 or 1 = through global memory (each sibling
                                           writes the parts other siblings own to its fp32
                                           buffer, keeps its own part in TMEM, and adds the
                                           others' parts from L2); 2 = through the owners' shared
                                           memory (distributed shared memory stores into a 64 KB
                                           receive buffer per CTA, which takes ring depth; needs
                                           tile_m * tile_n * 4 <= 65536, else UNSUPPORTED)       */
    int32_t split_clusters;             /* where the k-slices of a split tile run: 0 = library
                                           choice; 1 = in one cluster (the tile's CTAs are one
                                           cluster item); 2 = on separate clusters of a CTA pair
                                           each (every slice its own cluster item, partial sums
                                           exchanged through global memory with a per-tile count,
                                           in the same fixed order, so results are the same bits).
                                           2 needs MLP_MODE_PIPELINED, CTA pairs (cta_pair 0 or
                                           2), M <= 256 (one 256-row panel, so each stage
                                           boundary is one scoreboard group) and a grid with a
                                           cluster for every item of each split stage (a cluster
                                           then never holds two slices of one stage); else
                                           UNSUPPORTED                                           */
} mlp_chain_desc;

/* One record per tile of a pipelined run (MLP_DEBUG_EVENT_LOG), stage by stage, followed by one
 * record per CTA of the launch with stage = -1, tile = cta = the CTA index, t_start = kernel
 * entry, t_acc = set-up done (barriers, TMEM, cluster sync), t_end = exit.  t_* are %globaltimer ns;
 * seq_* come from one device-wide counter, taken after the consumer's acquire (start) and
 * before the producer's scoreboard release (end), so seq_end(p) < seq_start(c) for every
 * dependency p -> c.  In MLP_MODE_PIPELINED_KWAIT a consumer starts before its producers end
 * (it waits per k block), so start is when its CTA took the tile and that order need not hold. */
typedef struct {
    int32_t stage, tile, smid, cta;
    uint64_t t_start, t_end;
    uint32_t seq_start, seq_end;
    uint64_t t_acc;                     /* accumulator complete (split tiles: slice 0)           */
} mlp_event;

typedef struct {
    int32_t num_gemms;
    int32_t tile_m, tile_k;
    int32_t tile_n[MLP_MAX_GEMMS];
    int32_t tiles_m[MLP_MAX_GEMMS], tiles_n[MLP_MAX_GEMMS];
    int32_t grid_ctas;                  /* CTAs of the pipelined launch                          */
    int32_t num_sms;
    int32_t pipe_stages;                /* shared-memory ring depth                               */
    int32_t smem_bytes;                 /* dynamic shared memory per CTA                          */
    int32_t tmem_cols;
    int32_t launches_per_run;           /* kernels one mlp_chain_run enqueues                     */
    int32_t cluster_size;               /* CTAs per thread-block cluster                          */
    int32_t k_split[MLP_MAX_GEMMS];
    int32_t cta_pair;                   /* 2: CTA pairs (tile_m is then the pair's 256 rows)      */
    int32_t raster_group;               /* row panels per first-stage raster group (the caller's
                                           or the library's choice)                              */
    int32_t fill_k[MLP_MAX_GEMMS];      /* per GEMM: k depth of one ring fill (64 or 128);
                                           tile_k is the largest                                 */
    int32_t split_across[MLP_MAX_GEMMS]; /* per GEMM: 1 when its k-slices run on separate clusters
                                           (split_clusters)                                      */
    int32_t queue_free[MLP_MAX_GEMMS];  /* per stage boundary b (GEMM b -> b + 1), pipelined mode
                                           with the work-queue: 1 when its consumers skip the
                                           queue (one scoreboard group, or no more consumer
                                           items than co-resident clusters): consumer slot q
                                           takes the q-th member of the groups in group order
                                           and acquires its group's counter, and no release
                                           pushes; 0 when consumers poll queue entries           */
} mlp_chain_info;

typedef struct mlp_chain *mlp_chain_t;

/* Validate `desc`, build the dependency arrays, allocate the device state on desc->device.
 * On success *out owns everything it allocated.  Errors: INVALID_ARG, UNSUPPORTED, CUDA, OOM. */
mlp_status mlp_chain_create(const mlp_chain_desc *desc, mlp_chain_t *out);

/* Bytes of device workspace run() needs for the intermediates A_1 .. A_{S-1} (0 when S = 1). */
mlp_status mlp_chain_workspace_size(mlp_chain_t h, size_t *bytes);

/* Enqueue the whole chain on `stream` (asynchronous).  X: M x dims[0]; W[s]: dims[s] x
 * dims[s+1] (S + 1 weights when gated: see mlp_chain_desc.gated); Y: M x dims[S]; workspace:
 * >= mlp_chain_workspace_size bytes, 256-byte aligned.
 * All device pointers.  Returns INVALID_ARG for null or misaligned pointers, CUDA if a launch
 * fails, DEVICE_STATE if a previous device error has not been collected by mlp_chain_check. */
mlp_status mlp_chain_run(mlp_chain_t h, const void *X, const void *const *W, void *Y,
                         void *workspace, void *stream);

/* As mlp_chain_run, but X and Y are HOST buffers: enqueue the copy of X into the device
 * staging buffer X_dev, the chain, and the transfer of the result into Y_host, all on `stream`
 * (asynchronous; synchronise the stream before reading Y_host).  When Y_host is page-locked
 * memory the device can address (cudaHostAlloc, or cudaHostRegister with mapping; with unified
 * addressing every page-locked allocation qualifies, cudaPointerGetAttributes decides), the last
 * GEMM's epilogue stores its tiles straight into it as they complete, so the transfer overlaps the
 * chain and Y_dev is not written; otherwise Y_dev receives the result and is copied to Y_host. */
mlp_status mlp_chain_run_host(mlp_chain_t h, const void *X_host, const void *const *W,
                              void *Y_host, void *X_dev, void *Y_dev, void *workspace,
                              void *stream);

/* Synchronise `stream`, read the device status word and clear it.  Returns OK, TIMEOUT or
 * BAD_TILE; after a device error the handle's scoreboard, queues and tickets are re-initialised
 * so the next run starts clean.  The pages' consumer prologue polls the work-queue without a
 * limit (section III-A, Fig. 1; the polling CTA of section III-C, Fig. 2); here every such wait
 * has a deadline, because on one GPU nothing guarantees that the producer runs, and this call is
 * where a wait that ran out is reported (TIMEOUT) instead of hanging the device. */
mlp_status mlp_chain_check(mlp_chain_t h, void *stream);

/* The dependency array of stage boundary b (GEMM b produces, GEMM b+1 consumes), as host
 * arrays owned by the handle: prod_off[P+1], prod_tgt[prod_off[P]] (consumer ids ascending for
 * each producer), init_count[C].  Tile ids are row-major over each GEMM's tile grid.  This is the
 * host-built dependency array of section III-A (derived from the static dataflow of tiles: a
 * consumer tile reads one or more producer tiles); the pages leave its format open, and CSR by
 * producer plus an in-degree per consumer is this library's reading.  Valid until destroy. */
mlp_status mlp_chain_get_deps(mlp_chain_t h, int32_t boundary, const int32_t **prod_off,
                              const int32_t **prod_tgt, const int32_t **init_count,
                              int32_t *P, int32_t *C);

/* The scoreboard of one stage boundary: the counters the consumer prologue waits on (section
 * III-A, the scoreboard initialised from the dependency array).  Consumer tiles are partitioned
 * into groups that share one counter:
 *   - raster_group <= 1: a group is a class of consumer tiles with identical producer sets,
 *     numbered by its smallest member, members ascending (for a GEMM chain with equal row tiles:
 *     one row panel);
 *   - raster_group = g > 1: a group is the consumer tiles of g consecutive row panels (the last
 *     group may hold fewer), listed column by column, so its queue slots follow weight columns.
 * A group waits for grp_target = |union of its members' producer sets| x releases_per_producer
 * releases per run (each epilogue warp of each split-K slice of a producer tile releases once).
 * Every array is caller-owned and filled only when all six pointers are non-NULL; with any
 * pointer NULL only the five sizes are written (query them first).  Layout: int32, plain CSR:
 *   pg_off[producers + 1], pg_tgt[edges]   producer tile -> groups it feeds, ascending;
 *   grp_off[groups + 1],  grp_mem[consumers]  group -> member consumer tiles (push order);
 *   grp_target[groups];   cons_grp[consumers]  consumer tile -> its group. */
typedef struct {
    int32_t producers, consumers, groups, edges; /* sizes (written by the call)                 */
    int32_t releases_per_producer;               /* split-K slices x epilogue warps              */
    int32_t *pg_off, *pg_tgt, *grp_off, *grp_mem, *grp_target, *cons_grp;   /* caller buffers     */
} mlp_scoreboard;

/* Host-only scoreboard builder (no GPU needed), the routine mlp_chain_create uses: the groups of
 * the dependency array that mlp_deps_build gives for M x n_out producer tiles of bm x bn_p and
 * M x n_next consumer tiles of bm x bn_c.  Returns OK, or INVALID_ARG for a bad size or NULL sb. */
mlp_status mlp_scoreboard_build(int64_t M, int64_t n_out, int64_t n_next, int32_t bm, int32_t bn_p,
                                int32_t bn_c, int32_t raster_group, int32_t releases_per_producer,
                                mlp_scoreboard *sb);

/* The scoreboard tables the kernel of handle `h` waits on at stage boundary b, copied back from
 * the device (synchronous: waits for the device first) into sb's buffers; sizes as in
 * mlp_scoreboard_build.  INVALID_ARG for a bad boundary, CUDA if a copy fails. */
mlp_status mlp_chain_get_scoreboard(mlp_chain_t h, int32_t boundary, mlp_scoreboard *sb);

/* Copy the event log of the last pipelined run (synchronises the device) into host_buf, up to
 * cap records (tiles of all stages + CTAs of the launch); *n = records written.  INVALID_ARG without MLP_DEBUG_EVENT_LOG.  The records are
 * this library's form of the pages' per-phase timestamps (section III-C, Fig. 2: epilogue,
 * visibility, queue fetch and broadcast timed inside the kernels): globaltimer stamps at tile
 * start, accumulator complete and release, plus a device-wide sequence number for ordering. */
mlp_status mlp_chain_get_event_log(mlp_chain_t h, mlp_event *host_buf, size_t cap, size_t *n);

mlp_status mlp_chain_get_info(mlp_chain_t h, mlp_chain_info *info);

/* Free the handle and its device state (synchronises its internal streams). */
mlp_status mlp_chain_destroy(mlp_chain_t h);

/* Host-only dependency-array builder (no GPU needed), the same routine create() uses.
 * Producer tiles: bm_p x bn_p over an M x n_out output; consumer tiles: bm_c x bn_c over
 * M x n_next, each reading all n_out columns of its rows.  Pass NULL arrays to query sizes:
 * returns the number of edges (>= 0) or -1 on bad arguments / too small tgt_cap. */
int64_t mlp_deps_build(int64_t M, int64_t n_out, int64_t n_next, int32_t bm_p, int32_t bn_p,
                       int32_t bm_c, int32_t bn_c, int32_t *prod_off, int32_t *prod_tgt,
                       int64_t tgt_cap, int32_t *init_count);

/* Host model of the scoreboard / work-queue protocol (no GPU needed): `threads` host threads play
 * the persistent CTAs over a chain of `num_gemms` stages of tiles_m x tiles_n[s] tiles (consumers
 * read whole row panels) and run the kernel's protocol with its tables and its arithmetic
 * (protocol.h): first-stage raster and scoreboard groups of `raster_group` row panels (0 or 1:
 * none), releases_per_tile releases per finished tile (the kernel's split-K slices x epilogue
 * warps), counters that count up and accumulate over three back-to-back runs against the run's
 * epoch-scaled target, the completing release pushing the group's members column by column
 * (a boundary of one group, or of no more consumer tiles than threads, has no queue: consumer
 * slot q takes the q-th member of the groups in group order, as on the device),
 * relaxed queue polls followed by an acquire of the group counter before a consumer reads its
 * producers' output (plain reads: a missing happens-before edge is a data race for
 * ThreadSanitizer, a stale value fails the run), and seeded random delays.  order_out (optional,
 * one entry per tile of all stages) receives the first run's tiles in completion order as
 * stage << 24 | tile.  With drop_tile >= 0 that first-stage tile withholds its releases and the
 * run must end in MLP_ERR_TIMEOUT after timeout_ms.  Returns OK when every tile ran exactly once
 * per run after all of its producers and every counter ends each run exactly at its target. */
mlp_status mlp_protocol_model(int32_t num_gemms, int32_t tiles_m, const int32_t *tiles_n,
                              int32_t raster_group, int32_t releases_per_tile, int32_t threads,
                              uint64_t seed, int32_t drop_tile, uint32_t timeout_ms, int32_t *order_out);

/* As mlp_protocol_model, with k-slices on separate items (the kernel's split-K slices on separate
 * clusters of a CTA pair each, ChainDesc.split_clusters = 2).  slices (NULL: all 1) gives per stage
 * the number of slices S of each tile; S must divide releases_per_tile, and a stage with S > 1
 * must fit one wave: tiles_m * tiles_n[s] * S <= threads (siblings wait on one another).  Slice j
 * of a tile is the ticket after slice j-1 (first stage: the tile of raster position ticket / S;
 * later stages: work-queue slot ticket / S), makes releases_per_tile / S of the tile's releases
 * and, before them, exchanges partials with its siblings: each of its releases writes its own
 * partial and adds 1 to the tile's exchange counter, then the slice acquires that counter until it
 * reaches the run's target of releases_per_tile adds and reads its siblings' partials.  The
 * exchange counters accumulate over the three runs like the scoreboard's.  order_out (optional)
 * receives one entry per item, so a tile of a sliced stage appears S times.  drop_exchange >= 0
 * (a first-stage tile; the first stage must be sliced) makes that tile's last slice withhold its
 * exchange adds: the run must end in MLP_ERR_TIMEOUT.  Invalid sizes give MLP_ERR_INVALID_ARG. */
mlp_status mlp_protocol_model_slices(int32_t num_gemms, int32_t tiles_m, const int32_t *tiles_n,
                                     const int32_t *slices, int32_t raster_group, int32_t releases_per_tile,
                                     int32_t threads, uint64_t seed, int32_t drop_tile, int32_t drop_exchange,
                                     uint32_t timeout_ms, int32_t *order_out);

/* Allocation-free run of the two-GEMM chain (the paper has no counterpart to this entry point).
 *
 * For callers that cannot allocate device memory when they run the chain: code running inside
 * an allocator or memory-pool callback, runtimes that reserve all device memory up front and
 * forbid further cudaMalloc, or embeddings that must not go through the host framework's
 * caching allocator.  It needs no handle: it runs Y = (X*W1)*W2 (X: M x K, W1: K x N1,
 * W2: N1 x N2, Y: M x N2; bf16, device pointers, 16-byte aligned, K, N1, N2 multiples of 8) in
 * pipelined mode with the library's default tiles, and keeps every byte of scratch -- the
 * intermediate H, the dependency array, scoreboard, work-queue, tickets and status word -- in one
 * static device array of MLP_NOALLOC_SCRATCH_BYTES that each GPU loading the library holds until
 * the process exits.  It calls no cudaMalloc/cudaFree or other allocating routine.
 *   - Limit: shapes whose scratch (mainly M*N1*2 bytes of H) exceeds the array are rejected
 *     with MLP_ERR_INVALID_ARG before anything is enqueued.
 *   - The array and the kernel image are committed when the library's device code is loaded
 *     into a context: at the library's first CUDA call there, or, with lazy module loading (CUDA's
 *     default), possibly inside the first call of this entry point on that device.  So make one
 *     call (or create one handle) at start-up, outside any context that must not allocate, and
 *     before any stream capture; after that a call allocates nothing.
 *   - Each call looks up the array's device address and sets the kernel's shared-memory limit on
 *     the current device (both are per context, so a cudaDeviceReset needs nothing else).
 *   - Every call shares the one array: each call first re-initialises all of its state on
 *     `stream` (a small set-up kernel, then the chain kernel), so nothing of the previous call
 *     leaks in, but calls whose execution overlaps on the GPU (different streams, threads or
 *     processes sharing the device context) race and give wrong results.
 *   - With sync_check != 0 the call synchronises `stream` and returns MLP_ERR_TIMEOUT or
 *     MLP_ERR_BAD_TILE if the device reported one; with 0 it returns after enqueueing.  Pass 0
 *     while `stream` is being captured (a synchronisation would invalidate the capture). */
#define MLP_NOALLOC_SCRATCH_BYTES (16u << 20)
mlp_status mlp_chain_run_noalloc(int64_t M, int64_t K, int64_t N1, int64_t N2, const void *X,
                                 const void *W1, const void *W2, void *Y, int32_t sync_check,
                                 void *stream);

const char *mlp_status_str(mlp_status s);

#ifdef __cplusplus
}
#endif

#endif /* MLP_CHAIN_H_ */
