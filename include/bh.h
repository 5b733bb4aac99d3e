/*
 * bh.h -- C ABI of the GB300 Barnes-Hut gravity library (libbh.so).
 *
 * One call rebuilds an octree over N fp32 particles and returns, for every
 * particle (or for every point of a separate target set), the softened
 * acceleration and potential
 *
 *     a_i   = -G sum_j m_j (x_i - x_j) / (|x_i - x_j|^2 + eps^2)^{3/2}
 *     phi_i = -G sum_j m_j / (|x_i - x_j|^2 + eps^2)^{1/2}
 *
 * with a cell replaced by its centre of mass whenever w^2/theta^2 < r^2
 * (w = the cell's full edge, r = distance from the target to the cell's
 * centre of mass).  The pipeline and the opening test follow the GASPHiA
 * tree-code page ("GASPHiA中的自引力树代码效率与优化分析", sections
 * "计算核函数" and "性能瓶颈分析"); the build steps (bounding box, Morton
 * keys + spatial sort, octree) follow the tree page after Burtscher &
 * Pingali ("树结构（基于根据 Burtscher 和 Pingali 的研究）", section
 * "实现步骤").
 *
 * Conventions for every entry point:
 *  - All functions return an int status (BH_OK = 0, else a BH_E* code).
 *    bh_last_error() gives a one-line message for the last failure.
 *  - Particle arrays are AoS fp32 rows (x, y, z, m), 16 bytes per row, the
 *    base 16-byte aligned.  Result arrays are rows (ax, ay, az, phi).
 *  - "device" pointers are CUDA device (or managed) memory on the context's
 *    device; the caller owns them; the library never frees or retains them
 *    beyond the call's stream work.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device entry points only enqueue work: they return before the
 *    GPU finishes and perform no host synchronisation, except when a buffer
 *    must grow (documented at bh_compute).  Errors raised by kernels (a wait
 *    that timed out, a non-finite input) land in a device status word that
 *    bh_sync_status() reads.
 *  - A context is not thread-safe; use one context per host thread/stream.
 */
#ifndef BH_H
#define BH_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bh_ctx bh_ctx;

/* ---- status codes ---- */
#define BH_OK              0
#define BH_EINVAL          1   /* bad argument, or non-finite particle data  */
#define BH_ENOMEM          2   /* device or host allocation failed           */
#define BH_ECUDA           3   /* a CUDA runtime call or launch failed       */
#define BH_ETIMEOUT        4   /* a bounded device-side wait gave up         */
#define BH_ETREE_OVERFLOW  5   /* a node pool or traversal stack was too small */

/* ---- options for bh_set_option ---- */
#define BH_OPT_KEY_BITS      1  /* bits per axis of the Morton key: 21 (63-bit
                                   keys, default) or 10 (30-bit keys)        */
#define BH_OPT_LEAF_CAP      2  /* leaf capacity B in 1..64 (default 16): a
                                   cell is subdivided while it holds > B     */
#define BH_OPT_OPENING       3  /* group opening rule, see BH_OPEN_*         */
#define BH_OPT_TIMING        4  /* 1: record per-stage CUDA events (default 0) */
#define BH_OPT_GROUP         5  /* targets per warp group: 32, 64, or 0 (default):
                                   64, or 32 when the targets fill fewer groups
                                   of 64 than 16 per SM (below ~155k targets
                                   on 152 SMs) -- the opening vote is then
                                   taken over 32 targets                    */
#define BH_OPT_GRAPH         6  /* 1 (default): a call that repeats the previous
                                   one exactly (pointers, sizes, parameters,
                                   options) is captured once as a CUDA graph
                                   and replayed; 0: always launch kernels   */
#define BH_OPT_ESTIMATOR     7  /* BH_EST_* (default BH_EST_BARNES_HUT)       */
#define BH_OPT_SEED          8  /* stochastic estimator: 64-bit seed (default 0) */
#define BH_OPT_SAMPLES       9  /* stochastic estimator: paths per stratum,
                                   1..1024 (default 1)                       */
#define BH_OPT_PIPELINE     11  /* 1 (default): the group walk runs as
                                   producer/consumer warp pairs -- one warp
                                   traverses and fills list buffers, the
                                   other evaluates them (32 warps per SM);
                                   0: one warp does both for groups of 64
                                   (16 warps per SM); same results bit for
                                   bit.  Groups of 32 always run as pairs   */
#define BH_OPT_ORDER        12  /* spatial sort of sources and targets, see
                                   BH_ORDER_* (default BH_ORDER_RADIX)       */
#define BH_OPT_SHARDS       13  /* split the walk into this many shards,
                                   1..2^20 (default 1), see below            */
#define BH_OPT_SHARD        14  /* the shard the context's calls walk,
                                   0..shards-1 (default 0)                   */
#define BH_OPT_SCHEDULE     15  /* 1 (default): a call over the same groups
                                   as the previous call (same target count
                                   and group size, one shard, Barnes-Hut
                                   estimator) hands the groups to the walk
                                   heaviest first, by the terms each group
                                   evaluated in the previous call (two small
                                   extra kernels), when there are more
                                   groups than the walk takes at once (16 per
                                   SM); 2: whenever it can, even then; 0:
                                   Morton order.  The order changes no
                                   result, only how the walk's tail of long
                                   groups overlaps                           */
#define BH_OPT_TARGET_KEY_BITS 16 /* separate targets: bits per axis of the
                                   Morton key that orders them, 10 (30-bit
                                   keys, default: 4 radix passes) or 21.
                                   The order only decides which targets
                                   share a walk group; 2^10 cells per axis
                                   already separate any group of 64 that is
                                   spread over more than a 1/1024 of the
                                   targets' cube, and targets in one cell
                                   keep their input order               */
#define BH_OPT_STRATA_LEVEL 10  /* stochastic estimator: octree level s of the
                                   strata, 0..6 (default 2: up to 64 strata,
                                   the child count of the root of a tree with
                                   4 children per axis)                      */

/*
 * Spatial sort before the tree build (both give the same permutation, bit
 * for bit: stable by Morton key, ties by index).
 *
 * BH_ORDER_RADIX: least-significant-digit radix sort of (key, index), then a
 *   gather of the rows into key order.
 * BH_ORDER_TREE: the order of the GASPHiA tree-code page (section "排序算法"):
 *   an octree built by insertion (each row descends by octant, claims an
 *   empty child slot with atomicCAS or locks a slot holding another row and
 *   subdivides it until the two separate -- the tree page after Burtscher &
 *   Pingali, sections "构建树结构" and "基于稠密存储的并行树构建实现方案"),
 *   then subtree counts, and each parent hands its children consecutive
 *   ranges of the order from the top down.  Octants follow the Morton digits,
 *   then ten 3-bit digits of the row index, so the depth-first order is the
 *   (key, index) order.  Its node pool (80 bytes x (2 rows + 64), allocated
 *   at the first call that uses it) is enough for every measured workload
 *   (0.25-0.72 nodes per row); rows sharing very long digit prefixes can
 *   exhaust it, which bh_sync_status reports as BH_ETREE_OVERFLOW; the next
 *   call then gets a 4x larger pool (at most 32 nodes per row, which always
 *   suffices: the tree has at most 1 + 31 (rows - 1) nodes), so repeating
 *   the call succeeds.  Measured slower than BH_ORDER_RADIX on GB300; kept
 *   as the page's method.
 */
/*
 * Shards.  The walk visits the targets in Morton order, in groups (of
 * BH_OPT_GROUP targets; of 32 for the stochastic estimator).  With
 * BH_OPT_SHARDS = S and BH_OPT_SHARD = s, a call still builds the whole tree
 * and orders all targets, but walks only the groups [G s / S, G (s+1) / S)
 * (G = number of groups, integer division) and writes only those targets'
 * rows of acc_pot; the other rows are left as they were.  Every shard sees
 * the same tree and the same groups, so the rows written by shards 0..S-1 of
 * one input are the whole call's results bit for bit.  It is the split of
 * the work over GPUs with the sources (and targets) replicated, each GPU
 * walking one shard; the GASPHiA pages run on one GPU and have no such step.
 */
#define BH_ORDER_RADIX 0
#define BH_ORDER_TREE  1

#define BH_OPEN_VOTE  0  /* a cell is accepted for a group of targets only if
                            the opening test holds for every target of the
                            group (the page's __all_sync warp vote)          */
#define BH_OPEN_BOX   1  /* accepted if the test holds at the distance from
                            the centre of mass to the group's bounding box
                            (implies the vote, so more cells are opened).
                            For validation only: a group whose targets
                            straddle a high-level Morton boundary has a
                            large box and then walks most of the tree --
                            measured 4.8x (1M lattice) to 21x (5M galaxy)
                            slower than BH_OPEN_VOTE                        */

/*
 * Estimators of the traversal stage.  Both use the same tree.
 *
 * BH_EST_BARNES_HUT: the deterministic walk with the opening test and warp
 *   vote of the GASPHiA page (section "性能瓶颈分析").
 * BH_EST_STOCHASTIC: stochastic Barnes-Hut (page "Stochastic Barnes-Hut
 *   Approximation for Fast Summation on the GPU", section 方法, key designs
 *   1-4), an unbiased Monte Carlo estimate of the direct sum:
 *     F(q) = sum_R [ m_R f(p_R, q)
 *                    + (1/S) sum_samples sum_{surviving steps T}
 *                      Delta_T(q) (n_R / n_T) / P(reach T) ],
 *     Delta_T(q) = sum_{c child of T} m_c f(p_c, q) - m_T f(p_T, q),
 *   R over the strata (octree cells at level s and leaves above it), the
 *   path from R towards particle I (uniform among R's particles), each step
 *   surviving with probability min(1, max(1, b_T) / b_c), b = distance from
 *   the query to the centre of mass (to the particle, for a leaf's child)
 *   over the cell edge (half the leaf edge for a particle).  A leaf's children
 *   are its particles; in self mode the query's own particle contributes 0.
 *   Random numbers: Philox4x64-10 (Salmon et al., SC 2011), key (seed, 0),
 *   counter (group, stratum, sample, block): block 0 word 0 gives
 *   I = floor(word * n_R / 2^64), roulette step k uses block 1 + k/4 word
 *   k%4 as u = (word >> 40) * 2^-24.  With the child's edge w_T / 2,
 *   p = min(1, max(w_T, r_T) / (2 r_c)), and the step survives iff
 *   (4 (u u)) r_c^2 < max(w_T w_T, r_T^2) in fp32, every operation rounded
 *   as written.  A group is 32 consecutive queries in Morton order; its
 *   queries share every random number.  theta and BH_OPT_OPENING/GROUP do
 *   not apply.
 */
#define BH_EST_BARNES_HUT  0
#define BH_EST_STOCHASTIC  1

/* ---- debug knobs for bh_set_debug (tests only) ---- */
#define BH_DBG_SPIN_LIMIT  1    /* polls before a device wait gives up
                                   (default 1<<22); 0 makes every wait that
                                   is not already satisfied fail at once    */

/* ---- what bh_debug_export copies (after the stream's work is done) ---- */
#define BH_EXPORT_CUBE        1  /* float[4]: lo_x, lo_y, lo_z, L            */
#define BH_EXPORT_KEYS        2  /* uint64[n]: Morton keys in sorted order    */
#define BH_EXPORT_PERM        3  /* uint32[n]: perm[r] = caller index of the
                                    r-th particle in key order               */
#define BH_EXPORT_NODE_COUNT  4  /* int64[1]: number of tree nodes           */
#define BH_EXPORT_NODES       5  /* int32[6*nodes]: per node (level, first,
                                    count, first_child or -1, nchild, parent) */
#define BH_EXPORT_COM         6  /* float[4*nodes]: com x,y,z and mass       */
#define BH_EXPORT_TARGET_PERM 7  /* uint32[m]: Morton order of the targets   */
#define BH_EXPORT_WALK_STATS  8  /* uint64[4]: walk rounds, nodes tested,
                                    nodes decided by the vote, leaf chunks   */
#define BH_EXPORT_GROUP_COST  9  /* uint32[groups]: terms each walk group
                                    evaluated (targets x list entries), in
                                    group (Morton) order; BH_EINVAL unless
                                    the call recorded them (BH_OPT_SCHEDULE
                                    1, one shard, Barnes-Hut estimator)     */
#define BH_EXPORT_GROUP_ORDER 10 /* uint32[groups]: the order the call handed
                                    its groups to the walk; BH_EINVAL if it
                                    used Morton order                        */
#define BH_EXPORT_SORT_PATH   11 /* uint32[2]: 1 where the keys of the sources
                                    (then of separate targets) were sorted by
                                    the bucket path (63-bit keys, 4097 to
                                    256 * 4608 of them, every bucket of bits
                                    55..62 within 4608 keys: one pass on
                                    those bits, then each bucket sorted in
                                    shared memory), 0 where the digit passes
                                    ran; the permutation is the same        */

/* Stage indices for bh_get_stage_times. */
#define BH_STAGE_BBOX      0
#define BH_STAGE_KEYS      1
#define BH_STAGE_SORT      2
#define BH_STAGE_REORDER   3
#define BH_STAGE_BUILD     4
#define BH_STAGE_COM       5
#define BH_STAGE_TARGETS   6   /* bbox + keys + sort of a separate target set */
#define BH_STAGE_TRAVERSE  7   /* walk + write-back in caller order          */
#define BH_NUM_STAGES      8

/*
 * Create a context on CUDA device `device` with scratch for up to
 * `max_sources` particles and `max_targets` separate targets (either may be
 * 0; buffers grow on demand).  Defaults: theta 0.5, G 1, eps 0, options as
 * listed above.  *out is set to NULL on failure.  The GASPHiA page's code
 * allocates its device arrays in a class constructor (section "计算核函数",
 * the d_* arrays its kernels take); the context is that holder, in C form.
 */
int bh_create(bh_ctx **out, int device, size_t max_sources, size_t max_targets);

/* Destroy a context and free its scratch.  NULL is accepted.  No
 * counterpart in the pages (they free nothing explicitly). */
int bh_destroy(bh_ctx *c);

/*
 * Physical parameters: opening angle theta >= 0 (theta = 0 never accepts a
 * cell, reproducing the direct sum), gravitational constant G (finite), and
 * Plummer softening eps >= 0.  The GASPHiA page passes theta*theta and constG
 * to its gravity kernel (section "计算核函数"); the softening form is this
 * library's.  BH_EINVAL if out of range.
 */
int bh_set_params(bh_ctx *c, float theta, float G, float eps);

/* Set an option (BH_OPT_*).  BH_EINVAL for an unknown key or bad value.
 * Each option cites its passage above where the pages have one (key width
 * and spatial sort: the tree page's section "实现步骤"; the opening rule and
 * vote: the GASPHiA page's section "性能瓶颈分析"; the tree order: its
 * section "排序算法"); the rest (timing, graph replay, group size, pipeline,
 * shards, schedule) are this library's and have no counterpart. */
int bh_set_option(bh_ctx *c, int key, long long value);

/* Set a debug knob (BH_DBG_*); for tests of the failure paths.  No
 * counterpart in the pages. */
int bh_set_debug(bh_ctx *c, int key, long long value);

/*
 * Barnes-Hut gravity, the whole pipeline on `stream`: bounding cube ->
 * Morton keys -> radix sort + reorder -> octree build -> centre of mass ->
 * warp-cooperative walk -> results written back in caller order.
 *
 *   pos_mass  device, n rows (x,y,z,m) -- the sources.
 *   targets   device, m rows (x,y,z,*) or NULL.  NULL = self-gravity: the
 *             targets are the sources, each particle's own pair is skipped,
 *             and m is ignored.
 *   acc_pot   device, n (self) or m rows (ax,ay,az,phi), written in the same
 *             order as the particles/targets were given.
 *
 * n == 0 writes zeros for any targets and returns BH_OK.  If n (or m)
 * exceeds the context's capacity the scratch is reallocated first, which
 * synchronises the device once; all other calls are fully asynchronous and
 * can be captured in a CUDA graph.  Non-finite positions or masses set
 * BH_EINVAL in the device status word (results are then unspecified).
 *
 * Self mode with eps > 0: when a particle's own leaf is opened, its own
 * pair adds exactly m_i/eps to -phi_i and nothing to a_i, and the walk takes
 * it back out after the sum; the potential then carries an extra rounding
 * error of at most about k * 2^-24 * (m_i / eps) (k = terms evaluated for
 * the particle, typically 10^3), negligible unless eps is far below
 * m_i / |phi_i| (at the benchmark settings m_i/eps is 1e-4 of |phi_i| or
 * less).  bh_direct gives the own pair no term at all.
 */
int bh_compute(bh_ctx *c, const float *pos_mass, size_t n,
               const float *targets, size_t m, float *acc_pot, void *stream);

/*
 * Same as bh_compute with HOST buffers: copies the inputs to device staging
 * buffers owned by the context, computes, delivers the results and
 * synchronises `stream`.  Pinned (page-locked) host memory makes the copies
 * asynchronous DMA, and a pinned acc_pot is written by the kernels directly
 * (no copy back); pageable memory also works, through a staging buffer.
 * Returns the device status.
 */
int bh_compute_host(bh_ctx *c, const float *pos_mass, size_t n,
                    const float *targets, size_t m, float *acc_pot,
                    void *stream);

/*
 * Brute-force double loop (the GASPHiA page's 暴力双循环 reference, section
 * "精度与加速比验证"): every source acts on every target, sums kept in fp32
 * per tile of sources and in fp64 across tiles.  Same arguments and
 * conventions as bh_compute.
 */
int bh_direct(bh_ctx *c, const float *pos_mass, size_t n,
              const float *targets, size_t m, float *acc_pot, void *stream);

/*
 * Allocation-free brute-force sum, for callers that cannot allocate device
 * memory at the point where they need forces: code running while a CUDA
 * graph is being captured, loops that must never synchronise the device
 * (cudaMalloc/cudaFree may), and programs whose GPU memory is handed to
 * their own pool at start-up.  The pages have no counterpart of this entry
 * point; it is the bh_direct computation without a context.
 *
 *   pos_mass, targets, acc_pot: as in bh_direct (device, 16-byte aligned;
 *   targets NULL = self mode, own pair skipped).  G finite, eps >= 0.
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  Its only
 * scratch is a file-scope device array of 8 MiB (fp64 partial sums), held
 * by every GPU that loads the library until the process exits; at most
 * 262,144 targets per call (more returns BH_EINVAL).  It runs on the
 * current CUDA device, which must be the device of every pointer.  The
 * first call on a device looks up the array's device address (make it
 * before any stream capture) and keeps it for the life of the process; a
 * cudaDeviceReset of that device discards the array with the context, so
 * the kept address is then stale: do not call this entry point on a device
 * after the process has reset it.  Every call shares the one array, so
 * calls that overlap on the GPU (other streams, other host threads) race and
 * give wrong results; serialise them.  Returns BH_OK, BH_EINVAL (bad
 * pointer, alignment, parameter or size) or BH_ECUDA (a failed look-up or
 * launch of this call).
 */
int bh_direct_static(const float *pos_mass, size_t n, const float *targets,
                     size_t m, float G, float eps, float *acc_pot,
                     void *stream);

/*
 * Leapfrog (kick-drift-kick) time integration of a self-gravitating system
 * with the forces of bh_compute, the tree rebuilt from the new positions
 * every step -- the pure N-body run of the GASPHiA page (its galaxy-collision
 * video); the pages print no integrator, this is the plainest symplectic one:
 *     v += a dt/2;  x += v dt;  a = bh_compute(x);  v += a dt/2.
 *
 *   pos_mass  device, n rows (x,y,z,m); positions updated in place.
 *   vel       device, n rows (vx,vy,vz,unused); updated in place.
 *   acc_pot   device, n rows; with BH_LF_ACC_VALID in flags it must hold the
 *             accelerations at the initial positions (e.g. the output of the
 *             previous call), otherwise they are computed first.  On return
 *             it holds (ax,ay,az,phi) at the final positions.
 *   dt        time step (finite; negative runs backwards); nsteps >= 0.
 *
 * Asynchronous on `stream` like bh_compute; parameters and options are the
 * context's.  Errors of the device stages land in the status word.
 */
#define BH_LF_ACC_VALID 1
int bh_leapfrog(bh_ctx *c, float *pos_mass, float *vel, size_t n,
                float *acc_pot, float dt, int nsteps, int flags, void *stream);

/*
 * Synchronise `stream`, then return and clear the device status word
 * (BH_OK, BH_EINVAL for non-finite input, BH_ETIMEOUT, BH_ETREE_OVERFLOW).
 * The GASPHiA page checks every CUDA call and stops the program on an error
 * (its CUDA_CHECK macro, section "计算核函数"); here kernels record errors
 * in a status word instead, so the host learns of them without a fatal exit.
 */
int bh_sync_status(bh_ctx *c, void *stream);

/*
 * SPH neighbour search on the same octree ("树结构（基于根据 Burtscher 和
 * Pingali 的研究）" page, sections 粒子领域搜索 and 树遍历计算: the particles
 * within the kernel scale of each query, found by walking the tree; GASPHiA
 * keeps the per-node maximum smoothing length d_node_hmax for this search).
 * Particle j != i is a neighbour of i iff
 *     |x_i - x_j|^2 < (kappa H)^2,   H = max(h_i, h_j)  (BH_NB_SYMMETRIC)
 *                                    H = h_i            (BH_NB_GATHER)
 * with the test taken in fp32, every operation rounded as written:
 * d = x_i - x_j per axis, r2 = (dx dx + dy dy) + dz dz, s = kappa H,
 * neighbour iff r2 < s s.  The results are exact (no tolerance).
 *
 *   pos_mass  device, n rows (x,y,z,m); m is not used.
 *   h         device, n floats, smoothing lengths, finite and >= 0
 *             (otherwise the status word reads BH_EINVAL).
 *   kappa     kernel support in units of h (2 for the cubic spline), > 0.
 *   counts    device uint32[n], required: neighbours of particle i at i.
 *   offsets   device uint64[n+1] or NULL: exclusive scan of counts
 *             (offsets[n] = total).
 *   list      device uint32[list_cap] or NULL (needs offsets): particle i's
 *             neighbours (caller indices) at list[offsets[i] .. offsets[i+1]),
 *             in the walk's order (deterministic, not sorted).  Entries past
 *             list_cap are not written and the status word reads
 *             BH_ETREE_OVERFLOW; call once with list = NULL to size it.
 * Asynchronous on `stream` like bh_compute; it rebuilds the tree in the
 * context's scratch (BH_OPT_KEY_BITS and BH_OPT_LEAF_CAP apply) and replaces
 * the state bh_debug_export would read.  BH_EINVAL for bad arguments.
 */
#define BH_NB_GATHER     0
#define BH_NB_SYMMETRIC  1
int bh_neighbors(bh_ctx *c, const float *pos_mass, const float *h, size_t n,
                 float kappa, int mode, unsigned int *counts,
                 unsigned long long *offsets, unsigned int *list, size_t list_cap,
                 void *stream);

/*
 * fp32 throughput probe, for the roofline of the walk and direct-sum
 * kernels (bound by fp32 arithmetic); a calibration aid with no counterpart
 * in the pages.  Enqueues on `stream` one launch of a kernel whose threads
 * (2048 per SM) run 8 independent fused multiply-add chains for `iters`
 * steps, touching no memory: packed = 0 uses scalar fma.rn.f32, packed = 1
 * the packed fma.rn.f32x2 (two lane-FMAs per instruction).  `flops` (host,
 * or NULL) receives the fp32 flops of that launch, 2 per lane-FMA; time the
 * launch with events on `stream` and divide.  iters in 1..2^24, else
 * BH_EINVAL; BH_ECUDA if the launch fails.  Does not synchronise.
 */
int bh_fp32_probe(bh_ctx *c, int packed, int iters, double *flops, void *stream);

/*
 * Per-stage milliseconds of the last bh_compute made with BH_OPT_TIMING on
 * (indices BH_STAGE_*; a stage that did not run reads 0).  Synchronises on
 * the last recorded event.  n = number of floats at ms (<= BH_NUM_STAGES).
 * The stages are the GASPHiA page's timed kernels (section "性能测试与对比":
 * reset, bounding box, build, centre of mass, gravity), with the sort and
 * reorder of the tree page's section "实现步骤" timed on their own.
 */
int bh_get_stage_times(bh_ctx *c, float *ms, int n);

/*
 * Interaction counts of the last bh_compute (synchronises the device):
 * `executed` = source terms evaluated for valid targets by the group walk
 * (stochastic estimator: monopole evaluations, i.e. one per stratum plus,
 * per surviving step, the cell's children (or particles) and the cell);
 * `groups` = number of target groups walked.  After bh_neighbors,
 * `executed` = pair tests of its counting walk.
 * The "useful" count -- the terms of the per-target rule, the textbook
 * Barnes-Hut walk the GASPHiA page's section "性能瓶颈分析" starts from --
 * is not a by-product of the group walk: the group accepts a cell only when
 * all its targets do, so its terms are a superset and which of them a lone
 * target would have needed is never decided.  bh_count_interactions runs
 * that per-target walk separately (counting only, outside the step).
 */
int bh_get_counters(bh_ctx *c, unsigned long long *executed,
                    unsigned long long *groups);

/*
 * Per-target interaction count of the last bh_compute, on `stream`: for every
 * target, the number of terms (accepted cells + particle pairs, own pair
 * excluded) that a walk deciding the opening test per target -- the
 * textbook Barnes-Hut rule of the GASPHiA page's section "性能瓶颈分析"
 * without the warp vote -- evaluates on the same tree.  This is the minimum
 * work at this theta; the group walk of bh_compute evaluates a superset.
 * counts: device uint32[targets] in caller order, or NULL.  total: host, or
 * NULL; if given, `stream` is synchronised and the sum written.  The last
 * call's sources and targets must still be resident and unchanged.
 */
int bh_count_interactions(bh_ctx *c, unsigned int *counts,
                          unsigned long long *total, void *stream);

/*
 * Copy internal state of the last bh_compute to host memory (synchronises
 * the device).  `what` is a BH_EXPORT_* key; `bytes` is the size of
 * host_dst, which must hold the whole item (BH_EINVAL otherwise).  For the
 * bit-exact parity checks of keys, permutation and tree; no counterpart in
 * the pages.
 */
int bh_debug_export(bh_ctx *c, int what, void *host_dst, size_t bytes);

/* Message for the last failed call on this context ("" if none).  No
 * counterpart in the pages. */
const char *bh_last_error(const bh_ctx *c);

#ifdef __cplusplus
}
#endif

#endif /* BH_H */
