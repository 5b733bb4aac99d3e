/*
 * Barnes-Hut gravity oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what the GPU path
 * computes.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline may load it; the library never calls it.  It shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Sources (web pages this library implements):
 *   [T] "GASPHiA中的自引力树代码效率与优化分析" (yekq.top, GASPHiA tree code):
 *       sections "计算核函数" (the stages: bounding box, build, centre of mass,
 *       gravity), "性能瓶颈分析" (opening test w_sq/theta_sq < r_sq and the
 *       warp vote), "排序算法" (spatial sort), "精度与加速比验证" (brute force
 *       double loop as the accuracy reference).
 *   [S] "树结构（基于根据 Burtscher 和 Pingali 的研究）" (yekq.top, tree
 *       neighbour search): sections "实现步骤" (bounding box by reduction,
 *       Morton / Z-order keys and spatial sort), "构建树结构" (octant number
 *       x -> +1, y -> +2, z -> +4; subdivide until particles separate).
 *
 * Floating point: physics (centres of mass, forces, potentials) in fp64.  The
 * two integer-valued decisions the GPU takes in fp32 -- the bounding cube and
 * the Morton quantisation -- are taken here in fp32 with the same IEEE
 * operations (compile with -ffp-contract=off, no -ffast-math), as the pages
 * fix single precision for the particle data ([T] "性能测试与对比": 单精度).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - softening: a_i = -G sum m_j (x_i-x_j)/(|x_i-x_j|^2+eps^2)^{3/2},
 *    phi_i = -G sum m_j/(|x_i-x_j|^2+eps^2)^{1/2}; the pages give G only as a
 *    parameter and no eps.
 *  - cube anchored at the per-axis minimum lo with side L = max extent (1 if
 *    every point coincides); quantise q = trunc((x-lo)*(2^b/L)) clamped to
 *    [0, 2^b-1] -- a point on a split plane goes to the upper half.
 *  - w in the opening test is the full cell edge L/2^level; accept a cell iff
 *    w^2/theta^2 < r^2 (strict), r = distance from the target to the cell's
 *    centre of mass; the test applies to every cell, leaves included.
 *  - canonical octree with leaf capacity B: the root is level 0; a cell exists
 *    iff its parent is internal and some key lies in it; a cell is internal
 *    iff it holds more than B particles and its level is below b.
 *  - self mode skips the pair j == i by index; with eps == 0 a pair at zero
 *    separation contributes nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL 1

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Bounding cube ([S] 实现步骤 "确定粒子空间范围": min/max by reduction).        */
/* cube[0..2] = lo, cube[3] = L.  Returns ORC_EINVAL on NaN/Inf input.       */
/* ------------------------------------------------------------------------ */
int orc_bbox(const float *pm, int64_t n, float *cube)
{
    if (n <= 0) return ORC_EINVAL;
    float lo[3], hi[3];
    for (int a = 0; a < 3; ++a) { lo[a] = pm[a]; hi[a] = pm[a]; }
    for (int64_t i = 0; i < n; ++i) {
        for (int a = 0; a < 4; ++a)
            if (!isfinite(pm[4 * i + a])) return ORC_EINVAL;
        for (int a = 0; a < 3; ++a) {
            float v = pm[4 * i + a];
            if (v < lo[a]) lo[a] = v;
            if (v > hi[a]) hi[a] = v;
        }
    }
    float L = 0.0f;
    for (int a = 0; a < 3; ++a) {
        float e = hi[a] - lo[a];            /* fp32 subtraction */
        if (e > L) L = e;
    }
    if (L == 0.0f) L = 1.0f;
    for (int a = 0; a < 3; ++a) cube[a] = lo[a];
    cube[3] = L;
    return ORC_OK;
}

/* Quantise one coordinate to b bits on the cube (fp32, fixed op order). */
static uint32_t quantise(float x, float lo, float s, int bits)
{
    float v = (x - lo) * s;                 /* fp32 sub, then fp32 mul */
    float top = (float)((1u << bits) - 1u);
    if (!(v > 0.0f)) v = 0.0f;              /* also maps NaN (0*inf) to 0 */
    if (v > top) v = top;
    return (uint32_t)v;                     /* truncation toward zero */
}

void orc_quantise(const float *pm, int64_t n, const float *cube, int bits,
                  uint32_t *q)
{
    float s = (float)(1u << bits) / cube[3];   /* IEEE fp32 division */
    for (int64_t i = 0; i < n; ++i)
        for (int a = 0; a < 3; ++a)
            q[3 * i + a] = quantise(pm[4 * i + a], cube[a], s, bits);
}

/* Z-order interleave: bit k of qx -> key bit 3k, qy -> 3k+1, qz -> 3k+2, so
 * each 3-bit digit is the octant number x->1, y->2, z->4 of [S] 构建树结构. */
uint64_t orc_interleave(uint32_t qx, uint32_t qy, uint32_t qz, int bits)
{
    uint64_t key = 0;
    for (int k = 0; k < bits; ++k) {
        key |= (uint64_t)((qx >> k) & 1u) << (3 * k);
        key |= (uint64_t)((qy >> k) & 1u) << (3 * k + 1);
        key |= (uint64_t)((qz >> k) & 1u) << (3 * k + 2);
    }
    return key;
}

void orc_keys(const float *pm, int64_t n, const float *cube, int bits,
              uint64_t *keys)
{
    float s = (float)(1u << bits) / cube[3];
    for (int64_t i = 0; i < n; ++i) {
        uint32_t qx = quantise(pm[4 * i + 0], cube[0], s, bits);
        uint32_t qy = quantise(pm[4 * i + 1], cube[1], s, bits);
        uint32_t qz = quantise(pm[4 * i + 2], cube[2], s, bits);
        keys[i] = orc_interleave(qx, qy, qz, bits);
    }
}

/* ------------------------------------------------------------------------ */
/* Spatial sort ([S] 实现步骤 "粒子空间排序"): stable by key, ties by index.      */
/* ------------------------------------------------------------------------ */
typedef struct { uint64_t key; uint32_t idx; } kv_t;

static int kv_cmp(const void *a, const void *b)
{
    const kv_t *x = (const kv_t *)a, *y = (const kv_t *)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return x->idx < y->idx ? -1 : (x->idx > y->idx);
}

int orc_sort(const uint64_t *keys, int64_t n, uint32_t *perm)
{
    kv_t *t = (kv_t *)malloc(sizeof(kv_t) * (size_t)(n > 0 ? n : 1));
    if (!t) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) { t[i].key = keys[i]; t[i].idx = (uint32_t)i; }
    qsort(t, (size_t)n, sizeof(kv_t), kv_cmp);
    for (int64_t i = 0; i < n; ++i) perm[i] = t[i].idx;
    free(t);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Canonical octree over sorted keys, breadth first ([S] 构建树结构: a cell is  */
/* subdivided while it holds too many particles; children in octant order).  */
/* Node arrays: level, first (sorted index), count, child (index of the first */
/* child or -1), nchild.  Returns the node count, or -1 if cap is too small.  */
/* ------------------------------------------------------------------------ */
static int digit_at(uint64_t key, int level, int bits)
{
    /* 3-bit digit selecting the child at `level` (1..bits) */
    return (int)((key >> (3 * (bits - level))) & 7u);
}

int64_t orc_build_tree(const uint64_t *skeys, int64_t n, int bits, int leaf_cap,
                       int64_t cap, int32_t *level, int64_t *first,
                       int64_t *count, int64_t *child, int32_t *nchild)
{
    if (n <= 0) return 0;
    if (cap < 1) return -1;
    int64_t head = 0, tail = 0;
    level[tail] = 0; first[tail] = 0; count[tail] = n;
    child[tail] = -1; nchild[tail] = 0; ++tail;
    while (head < tail) {                   /* queue order = breadth first */
        int64_t c = head++;
        int l = level[c];
        if (!(count[c] > leaf_cap && l < bits)) continue;   /* leaf */
        int64_t s = first[c], e = first[c] + count[c];
        child[c] = tail;
        int64_t run = s;
        while (run < e) {
            int d = digit_at(skeys[run], l + 1, bits);
            int64_t r = run;
            while (r < e && digit_at(skeys[r], l + 1, bits) == d) ++r;
            if (tail >= cap) return -1;
            level[tail] = l + 1; first[tail] = run; count[tail] = r - run;
            child[tail] = -1; nchild[tail] = 0; ++tail;
            nchild[c] += 1;
            run = r;
        }
    }
    return tail;
}

/* ------------------------------------------------------------------------ */
/* Centre of mass per node ([T] 计算节点质心), fp64 sums over each node's      */
/* sorted particle range.  A massless node sits at its cell centre.           */
/* com[4*c..] = (x, y, z, mass).                                              */
/* ------------------------------------------------------------------------ */
static uint32_t deinterleave(uint64_t key, int axis, int bits)
{
    uint32_t q = 0;
    for (int k = 0; k < bits; ++k)
        q |= (uint32_t)((key >> (3 * k + axis)) & 1u) << k;
    return q;
}

void orc_com(const float *spm, const uint64_t *skeys, int64_t nnodes,
             const int32_t *level, const int64_t *first, const int64_t *count,
             const float *cube, int bits, double *com)
{
    double L = cube[3];
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t c = 0; c < nnodes; ++c) {
        double m = 0.0, sx = 0.0, sy = 0.0, sz = 0.0;
        for (int64_t j = first[c]; j < first[c] + count[c]; ++j) {
            double mj = spm[4 * j + 3];
            m += mj;
            sx += mj * (double)spm[4 * j + 0];
            sy += mj * (double)spm[4 * j + 1];
            sz += mj * (double)spm[4 * j + 2];
        }
        if (m != 0.0) {
            com[4 * c + 0] = sx / m; com[4 * c + 1] = sy / m; com[4 * c + 2] = sz / m;
        } else {
            double w = ldexp(L, -level[c]);
            int sh = bits - level[c];
            for (int a = 0; a < 3; ++a) {
                uint32_t cell = deinterleave(skeys[first[c]], a, bits) >> sh;
                com[4 * c + a] = (double)cube[a] + ((double)cell + 0.5) * w;
            }
        }
        com[4 * c + 3] = m;
    }
}

/* ------------------------------------------------------------------------ */
/* One softened pair term, source (sx,sy,sz,m) acting on target x.           */
/* ------------------------------------------------------------------------ */
static inline void pair_term(const double *x, double sx, double sy, double sz,
                             double m, double eps2, double *acc)
{
    double dx = sx - x[0], dy = sy - x[1], dz = sz - x[2];
    double r2 = dx * dx + dy * dy + dz * dz + eps2;
    if (r2 == 0.0) return;                  /* eps == 0 and coincident */
    double inv = 1.0 / sqrt(r2);
    double inv3 = inv * inv * inv;
    acc[0] += m * dx * inv3;
    acc[1] += m * dy * inv3;
    acc[2] += m * dz * inv3;
    acc[3] -= m * inv;
}

/* Magnitude of the acceleration term of one pair (for error scales). */
static inline double pair_mag(const double *x, double sx, double sy, double sz,
                              double m, double eps2)
{
    double dx = sx - x[0], dy = sy - x[1], dz = sz - x[2];
    double r2 = dx * dx + dy * dy + dz * dz + eps2;
    if (r2 == 0.0) return 0.0;
    return fabs(m) * sqrt(dx * dx + dy * dy + dz * dz) / (r2 * sqrt(r2));
}

/* ------------------------------------------------------------------------ */
/* Brute-force double loop ([T] 精度与加速比验证: 暴力计算 reference).           */
/* tgt == NULL: self mode over the sources (pair j == i skipped).            */
/* idx (may be NULL): evaluate only targets idx[0..k-1]; out has k rows.     */
/* ------------------------------------------------------------------------ */
void orc_direct(const float *src, int64_t n, const float *tgt, int64_t m,
                const int64_t *idx, int64_t k, double G, double eps,
                double *out)
{
    int self = (tgt == NULL);
    const float *T = self ? src : tgt;
    int64_t cnt = idx ? k : (self ? n : m);
    double eps2 = eps * eps;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < cnt; ++r) {
        int64_t i = idx ? idx[r] : r;
        double x[3] = {T[4 * i], T[4 * i + 1], T[4 * i + 2]};
        double acc[4] = {0, 0, 0, 0};
        for (int64_t j = 0; j < n; ++j) {
            if (self && j == i) continue;
            pair_term(x, src[4 * j], src[4 * j + 1], src[4 * j + 2],
                      src[4 * j + 3], eps2, acc);
        }
        for (int a = 0; a < 4; ++a) out[4 * r + a] = G * acc[a];
    }
}

/* ------------------------------------------------------------------------ */
/* Barnes-Hut walk for one target ([T] 性能瓶颈分析: accept a cell iff          */
/* w_sq/theta_sq < r_sq, otherwise open it; particles are always exact).      */
/* self_j: sorted index of the target's own particle, or -1.                 */
/* Returns the number of terms (accepted cells + particle pairs).            */
/* ------------------------------------------------------------------------ */
typedef struct {
    const float *spm;        /* sorted sources (x,y,z,m) */
    int64_t nnodes;
    const int32_t *level;
    const int64_t *first, *count, *child;
    const int32_t *nchild;
    const double *com;       /* (x,y,z,m) per node */
    double L, theta, eps2;
} tree_t;

static int64_t walk_one(const tree_t *t, const double *x, int64_t self_j,
                        double *acc, int64_t *stack)
{
    double th2 = t->theta * t->theta;
    int64_t terms = 0, sp = 0;
    stack[sp++] = 0;
    while (sp > 0) {
        int64_t c = stack[--sp];
        double w = ldexp(t->L, -t->level[c]);
        const double *cm = t->com + 4 * c;
        double dx = cm[0] - x[0], dy = cm[1] - x[1], dz = cm[2] - x[2];
        double r2 = dx * dx + dy * dy + dz * dz;
        if ((w * w) / th2 < r2) {           /* accept the cell as one mass */
            pair_term(x, cm[0], cm[1], cm[2], cm[3], t->eps2, acc);
            ++terms;
        } else if (t->child[c] < 0) {       /* leaf: its particles, exactly */
            for (int64_t j = t->first[c]; j < t->first[c] + t->count[c]; ++j) {
                if (j == self_j) continue;
                const float *p = t->spm + 4 * j;
                pair_term(x, p[0], p[1], p[2], p[3], t->eps2, acc);
                ++terms;
            }
        } else {                            /* open: visit children in order */
            for (int k = t->nchild[c] - 1; k >= 0; --k)
                stack[sp++] = t->child[c] + k;
        }
    }
    return terms;
}

/* Per-target Barnes-Hut.  tgt_pos: k target points (x,y,z,*) as fp32 rows;
 * self_j: k sorted self indices or NULL.  out: k rows (ax,ay,az,phi)*G. */
void orc_bh(const float *spm, int64_t nnodes, const int32_t *level,
            const int64_t *first, const int64_t *count, const int64_t *child,
            const int32_t *nchild, const double *com, double L, double theta,
            double G, double eps, const float *tgt_pos, const int64_t *self_j,
            int64_t k, double *out, int64_t *terms)
{
    tree_t t = {spm, nnodes, level, first, count, child, nchild, com, L, theta,
                eps * eps};
#pragma omp parallel
    {
        int64_t *stack = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nnodes + 8));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < k; ++r) {
            double x[3] = {tgt_pos[4 * r], tgt_pos[4 * r + 1], tgt_pos[4 * r + 2]};
            double acc[4] = {0, 0, 0, 0};
            int64_t nt = walk_one(&t, x, self_j ? self_j[r] : -1, acc, stack);
            for (int a = 0; a < 4; ++a) out[4 * r + a] = G * acc[a];
            if (terms) terms[r] = nt;
        }
        free(stack);
    }
}

/* ------------------------------------------------------------------------ */
/* Group walk: the warp-vote form of [T] 性能瓶颈分析.  A group of consecutive */
/* targets walks the tree together; a cell is accepted only if the test      */
/* holds for every target of the group (mode 0: per-target vote, the page's  */
/* __all_sync), or if it holds for the distance from the centre of mass to   */
/* the group's bounding box (mode 1: box test, which implies mode 0).        */
/* Every accepted cell and every particle of an opened leaf is applied to    */
/* every target of the group.  Targets are given in group order.  absacc     */
/* (may be NULL) receives, per target, G * sum |acceleration term|: the scale */
/* of the rounding error of any summation of the same terms.                 */
/* ------------------------------------------------------------------------ */
void orc_bh_group(const float *spm, int64_t nnodes, const int32_t *level,
                  const int64_t *first, const int64_t *count,
                  const int64_t *child, const int32_t *nchild,
                  const double *com, double L, double theta, double G,
                  double eps, const float *tgt_pos, const int64_t *self_j,
                  int64_t k, int64_t group, int mode, double *out,
                  int64_t *terms, double *absacc)
{
    double th2 = theta * theta, eps2 = eps * eps;
    int64_t ngroups = (k + group - 1) / group;
#pragma omp parallel
    {
        int64_t *stack = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nnodes + 8));
        double *acc = (double *)malloc(sizeof(double) * 5 * (size_t)group);
#pragma omp for schedule(dynamic, 4)
        for (int64_t g = 0; g < ngroups; ++g) {
            int64_t t0 = g * group, t1 = t0 + group < k ? t0 + group : k;
            double blo[3] = {INFINITY, INFINITY, INFINITY};
            double bhi[3] = {-INFINITY, -INFINITY, -INFINITY};
            for (int64_t r = t0; r < t1; ++r)
                for (int a = 0; a < 3; ++a) {
                    double v = tgt_pos[4 * r + a];
                    if (v < blo[a]) blo[a] = v;
                    if (v > bhi[a]) bhi[a] = v;
                }
            memset(acc, 0, sizeof(double) * 5 * (size_t)group);
            double *mag = acc + 4 * (size_t)group;
            int64_t nterm = 0, sp = 0;
            stack[sp++] = 0;
            while (sp > 0) {
                int64_t c = stack[--sp];
                double w = ldexp(L, -level[c]);
                double ropen2 = (w * w) / th2;
                const double *cm = com + 4 * c;
                int accept = 1;
                if (mode == 0) {
                    for (int64_t r = t0; r < t1 && accept; ++r) {
                        double dx = cm[0] - tgt_pos[4 * r];
                        double dy = cm[1] - tgt_pos[4 * r + 1];
                        double dz = cm[2] - tgt_pos[4 * r + 2];
                        if (!(ropen2 < dx * dx + dy * dy + dz * dz)) accept = 0;
                    }
                } else {
                    double d2 = 0.0;
                    for (int a = 0; a < 3; ++a) {
                        double d = 0.0;
                        if (cm[a] < blo[a]) d = blo[a] - cm[a];
                        else if (cm[a] > bhi[a]) d = cm[a] - bhi[a];
                        d2 += d * d;
                    }
                    accept = ropen2 < d2;
                }
                if (accept) {
                    for (int64_t r = t0; r < t1; ++r) {
                        double x[3] = {tgt_pos[4 * r], tgt_pos[4 * r + 1], tgt_pos[4 * r + 2]};
                        pair_term(x, cm[0], cm[1], cm[2], cm[3], eps2, acc + 4 * (r - t0));
                        mag[r - t0] += pair_mag(x, cm[0], cm[1], cm[2], cm[3], eps2);
                    }
                    nterm += t1 - t0;
                } else if (child[c] < 0) {
                    for (int64_t j = first[c]; j < first[c] + count[c]; ++j) {
                        const float *p = spm + 4 * j;
                        for (int64_t r = t0; r < t1; ++r) {
                            if (self_j && self_j[r] == j) continue;
                            double x[3] = {tgt_pos[4 * r], tgt_pos[4 * r + 1], tgt_pos[4 * r + 2]};
                            pair_term(x, p[0], p[1], p[2], p[3], eps2, acc + 4 * (r - t0));
                            mag[r - t0] += pair_mag(x, p[0], p[1], p[2], p[3], eps2);
                        }
                    }
                    nterm += count[c] * (t1 - t0);
                } else {
                    for (int q = nchild[c] - 1; q >= 0; --q)
                        stack[sp++] = child[c] + q;
                }
            }
            for (int64_t r = t0; r < t1; ++r) {
                for (int a = 0; a < 4; ++a) out[4 * r + a] = G * acc[4 * (r - t0) + a];
                if (absacc) absacc[r] = fabs(G) * mag[r - t0];
            }
            if (terms) terms[g] = nterm;
        }
        free(acc);
        free(stack);
    }
}

/* ------------------------------------------------------------------------ */
/* Leapfrog time integration, kick-drift-kick, with brute-force forces      */
/* ([T] title video: the 5M-particle galaxy collision is a pure N-body run   */
/* advanced step by step; the pages do not print an integrator, so the      */
/* plainest symplectic one is used).  One step:                             */
/*   v += a(x) dt/2;  x += v dt;  v += a(x) dt/2.                            */
/* pos (x,y,z,m) and vel (vx,vy,vz) are fp64, updated in place.              */
/* ------------------------------------------------------------------------ */
static void accel64(const double *pos, int64_t n, double G, double eps2,
                    double *acc)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double a[3] = {0, 0, 0};
        for (int64_t j = 0; j < n; ++j) {
            if (j == i) continue;
            double dx = pos[4 * j] - pos[4 * i];
            double dy = pos[4 * j + 1] - pos[4 * i + 1];
            double dz = pos[4 * j + 2] - pos[4 * i + 2];
            double r2 = dx * dx + dy * dy + dz * dz + eps2;
            if (r2 == 0.0) continue;
            double inv = 1.0 / sqrt(r2);
            double w = pos[4 * j + 3] * inv * inv * inv;
            a[0] += w * dx; a[1] += w * dy; a[2] += w * dz;
        }
        for (int k = 0; k < 3; ++k) acc[3 * i + k] = G * a[k];
    }
}

void orc_leapfrog(double *pos, double *vel, int64_t n, double G, double eps,
                  double dt, int64_t nsteps)
{
    double *acc = (double *)malloc(sizeof(double) * 3 * (size_t)(n > 0 ? n : 1));
    double eps2 = eps * eps;
    accel64(pos, n, G, eps2, acc);
    for (int64_t s = 0; s < nsteps; ++s) {
        for (int64_t i = 0; i < n; ++i)
            for (int k = 0; k < 3; ++k) {
                vel[3 * i + k] += 0.5 * dt * acc[3 * i + k];
                pos[4 * i + k] += dt * vel[3 * i + k];
            }
        accel64(pos, n, G, eps2, acc);
        for (int64_t i = 0; i < n; ++i)
            for (int k = 0; k < 3; ++k) vel[3 * i + k] += 0.5 * dt * acc[3 * i + k];
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* Philox4x64-10, the counter-based generator of Salmon, Moraes, Dror and    */
/* Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011).  Each of   */
/* ten rounds forms the 128-bit products of words 0 and 2 with the two round */
/* multipliers, builds the new words from the high halves xor the odd words  */
/* xor the key and from the low halves, then adds the two Weyl constants to  */
/* the key.                                                                  */
/* ------------------------------------------------------------------------ */
void orc_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        unsigned __int128 p0 = (unsigned __int128)0xD2E7470EE14C6C93ull * x0;
        unsigned __int128 p1 = (unsigned __int128)0xCA5A826395121157ull * x2;
        uint64_t y0 = (uint64_t)(p1 >> 64) ^ x1 ^ k0;
        uint64_t y1 = (uint64_t)p1;
        uint64_t y2 = (uint64_t)(p0 >> 64) ^ x3 ^ k1;
        uint64_t y3 = (uint64_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* ------------------------------------------------------------------------ */
/* Stochastic Barnes-Hut ([P] "Stochastic Barnes-Hut Approximation for Fast  */
/* Summation on the GPU", section 方法, 关键设计 1-4).  The exact sum is a     */
/* telescoping sum along each source's root-to-leaf path; one path per       */
/* stratum is drawn (index I uniform among the stratum's particles), its     */
/* length cut by Russian roulette, and each refinement step that survives is */
/* weighted by 1 / (P(I in T) * P(reach the step)), which keeps the estimate  */
/* unbiased.  Refining a cell T replaces its monopole by its children's:     */
/*   Delta_T(q) = sum_{c child of T} m_c f(p_c, q) - m_T f(p_T, q)            */
/* Readings where the page is silent or written for another tree:            */
/*  - tree: the canonical octree above (2 children per axis, not the page's  */
/*    4); strata are its cells at level s plus the leaves above level s,     */
/*    standing in for the children of the page's root;                       */
/*  - a leaf's children are its particles (the self particle contributes 0);*/
/*    a particle's size is half the edge of its leaf;                       */
/*  - far-field ratio beta(T) = |q - p_T| / w_T, p_T the centre of mass, w_T */
/*    the cell edge; continue from T to the path child c with probability   */
/*    p = min(1, max(1, beta(T)) / beta(c)), 1 where beta(c) = 0.  The child */
/*    edge is w_T / 2 (a cell's or a particle's), so p = min(1, max(w_T,     */
/*    r_T) / (2 r_c)), r = distance to the centre of mass (the particle).    */
/*    The decision u < p is taken in fp32 (the page computes in single       */
/*    precision) on squares, with every operation rounded as written:       */
/*    (4 (u u)) r_c^2 < max(w_T w_T, r_T^2); everything else in fp64;       */
/*  - random numbers: Philox4x64-10, key (seed, 0), counter (group, stratum, */
/*    sample, block).  Block 0 word 0 gives I = floor(o * n_R / 2^64);       */
/*    roulette step k uses block 1 + k/4, word k%4, as u = (o >> 40) 2^-24.  */
/*    Queries of one group (32 consecutive Morton-ordered queries, one warp) */
/*    share every random number, as the page shares seeds across a warp;     */
/*  - S samples per stratum are averaged.                                    */
/* grp[r]: group of target row r.  out: k rows (ax,ay,az,phi)*G.  terms:     */
/* kernel evaluations per row.  scale (may be NULL): k rows of four error    */
/* scales, each times |G|: sum |weight * term| of the acceleration and of the */
/* potential (the scale of summation rounding), and sum over cell terms of   */
/* |weight| m / (r^2+eps^2)^{3/2} and |weight| m r / (r^2+eps^2)^{3/2}, the   */
/* sensitivity of the acceleration and of the potential to a displacement of */
/* the cells' centres of mass (which an fp32 implementation rounds).         */
/* ------------------------------------------------------------------------ */
/* squared distance in fp32, rounded in this order */
static float dist2_32(const float *q, const float *p)
{
    float dx = q[0] - p[0], dy = q[1] - p[1], dz = q[2] - p[2];
    float d2 = dx * dx + dy * dy;
    return d2 + dz * dz;
}

/* the roulette: does the step from T to its path child survive draw u? */
static int survives(float u, float wT, float dT2, float dc2)
{
    float lhs = (4.0f * (u * u)) * dc2;
    float rhs = fmaxf(wT * wT, dT2);
    return lhs < rhs;
}

/* the survival probability of that step, for the weight (fp64) */
static double survival_prob(float wT, float dT2, float dc2)
{
    if (!(dc2 > 0.0f)) return 1.0;
    double rhs = fmax((double)wT * (double)wT, (double)dT2);
    double p = sqrt(rhs / (4.0 * (double)dc2));
    return p < 1.0 ? p : 1.0;
}

/* one weighted softened term of mass m at s on target x; sc accumulates the */
/* four error scales (the last two only for cells, cell != 0)                */
static int64_t wterm(const double *x, double sx, double sy, double sz, double m,
                     double wgt, double eps2, int cell, double *acc, double *sc)
{
    double t[4] = {0, 0, 0, 0};
    pair_term(x, sx, sy, sz, m, eps2, t);
    for (int a = 0; a < 4; ++a) acc[a] += wgt * t[a];
    sc[0] += fabs(wgt) * pair_mag(x, sx, sy, sz, m, eps2);
    sc[1] += fabs(wgt * t[3]);
    if (cell) {
        double dx = sx - x[0], dy = sy - x[1], dz = sz - x[2];
        double r2 = dx * dx + dy * dy + dz * dz;
        double s2 = r2 + eps2;
        if (s2 > 0.0) {
            sc[2] += fabs(wgt * m) / (s2 * sqrt(s2));
            sc[3] += fabs(wgt * m) * sqrt(r2) / (s2 * sqrt(s2));
        }
    }
    return 1;
}

void orc_sbh(const float *spm, int64_t nnodes, const int32_t *level,
             const int64_t *first, const int64_t *count, const int64_t *child,
             const int32_t *nchild, const double *com, float L, double G,
             double eps, const float *tgt_pos, const int64_t *self_j,
             const int64_t *grp, int64_t k, uint64_t seed, int strata_level,
             int samples, double *out, int64_t *terms, double *scale)
{
    double eps2 = eps * eps;
    /* strata, in node order */
    int64_t ns = 0;
    int64_t *strata = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nnodes + 1));
    for (int64_t c = 0; c < nnodes; ++c)
        if (level[c] == strata_level || (level[c] < strata_level && child[c] < 0))
            strata[ns++] = c;
    const uint64_t key[2] = {seed, 0};
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < k; ++r) {
        const float qf[3] = {tgt_pos[4 * r], tgt_pos[4 * r + 1], tgt_pos[4 * r + 2]};
        const double x[3] = {qf[0], qf[1], qf[2]};
        const int64_t self = self_j ? self_j[r] : -1;
        double acc[4] = {0, 0, 0, 0}, sc[4] = {0, 0, 0, 0};
        int64_t nterm = 0;
        for (int64_t si = 0; si < ns; ++si) {
            const int64_t R = strata[si];
            const double *cR = com + 4 * R;
            /* the stratum's monopole */
            nterm += wterm(x, cR[0], cR[1], cR[2], cR[3], 1.0, eps2, 1, acc, sc);
            for (int s = 0; s < samples; ++s) {
                uint64_t ctr[4] = {(uint64_t)grp[r], (uint64_t)si, (uint64_t)s, 0};
                uint64_t o[4], ou[4];
                orc_philox4x64(ctr, key, o);
                int64_t I = (int64_t)(((unsigned __int128)o[0] *
                                       (unsigned __int128)(uint64_t)count[R]) >> 64);
                int64_t J = first[R] + I;        /* sorted index of the path's particle */
                int64_t T = R;
                double P = 1.0;
                for (int step = 0;; ++step) {
                    const int leaf = child[T] < 0;
                    const float wT = ldexpf(L, -level[T]);
                    const float pT[3] = {(float)com[4 * T], (float)com[4 * T + 1],
                                         (float)com[4 * T + 2]};
                    int64_t c = -1;              /* path child node (internal T) */
                    float pc[3];
                    if (leaf) {
                        for (int a = 0; a < 3; ++a) pc[a] = spm[4 * J + a];
                    } else {
                        for (int q = 0; q < nchild[T]; ++q) {
                            int64_t cc = child[T] + q;
                            if (first[cc] <= J && J < first[cc] + count[cc]) c = cc;
                        }
                        for (int a = 0; a < 3; ++a) pc[a] = (float)com[4 * c + a];
                    }
                    const float dT2 = dist2_32(qf, pT), dc2 = dist2_32(qf, pc);
                    if (step % 4 == 0) {
                        ctr[3] = (uint64_t)(1 + step / 4);
                        orc_philox4x64(ctr, key, ou);
                    }
                    float u = (float)(ou[step % 4] >> 40) * 0x1p-24f;
                    if (!survives(u, wT, dT2, dc2)) break;   /* roulette ends the path */
                    P *= survival_prob(wT, dT2, dc2);
                    double wgt = ((double)count[R] / (double)count[T]) / P / samples;
                    /* Delta_T: children's monopoles minus T's own */
                    if (leaf) {
                        for (int64_t j = first[T]; j < first[T] + count[T]; ++j) {
                            if (j == self) continue;
                            const float *pj = spm + 4 * j;
                            nterm += wterm(x, pj[0], pj[1], pj[2], pj[3], wgt, eps2,
                                           0, acc, sc);
                        }
                    } else {
                        for (int q = 0; q < nchild[T]; ++q) {
                            const double *cc = com + 4 * (child[T] + q);
                            nterm += wterm(x, cc[0], cc[1], cc[2], cc[3], wgt, eps2,
                                           1, acc, sc);
                        }
                    }
                    const double *cT = com + 4 * T;
                    nterm += wterm(x, cT[0], cT[1], cT[2], cT[3], -wgt, eps2, 1,
                                   acc, sc);
                    if (leaf) break;
                    T = c;
                }
            }
        }
        for (int a = 0; a < 4; ++a) out[4 * r + a] = G * acc[a];
        if (terms) terms[r] = nterm;
        if (scale)
            for (int a = 0; a < 4; ++a) scale[4 * r + a] = fabs(G) * sc[a];
    }
    free(strata);
}

/* ------------------------------------------------------------------------ */
/* SPH neighbour search ([S] "树结构（基于根据 Burtscher 和 Pingali 的研究）", */
/* sections 1 粒子领域搜索 and 实现步骤 / 树遍历计算: find the particles within */
/* the kernel scale of each query; [T] GASPHiA keeps a per-node maximum      */
/* smoothing length, d_node_hmax, for that search).  The definition written */
/* out: particle j != i is a neighbour of i iff                              */
/*   |x_i - x_j|^2 < (kappa * H)^2,  H = max(h_i, h_j)  (mode 1, symmetric)  */
/*                                   H = h_i            (mode 0, gather)    */
/* Readings: kappa is the kernel's support in units of h; the test is taken  */
/* in fp32 (the pages' particle data are single precision) with every       */
/* operation rounded as written: d = x_i - x_j per axis,                    */
/* r2 = (dx dx + dy dy) + dz dz, s = kappa H, s2 = s s, neighbour iff       */
/* r2 < s2.  Brute force over all pairs, no tree.                           */
/* rows: the k query rows (indices into pm); counts[r]: neighbours of row   */
/* r; list (may be NULL): row r's neighbours in ascending index order at    */
/* list[offs[r] ..], offs (k+1 entries) given by the caller.                */
/* ------------------------------------------------------------------------ */
static int is_neighbour(const float *pm, const float *h, int64_t i, int64_t j,
                        float kappa, int mode)
{
    float dx = pm[4 * i] - pm[4 * j];
    float dy = pm[4 * i + 1] - pm[4 * j + 1];
    float dz = pm[4 * i + 2] - pm[4 * j + 2];
    float r2 = dx * dx + dy * dy;
    r2 = r2 + dz * dz;
    float H = mode == 1 ? fmaxf(h[i], h[j]) : h[i];
    float s = kappa * H;
    float s2 = s * s;
    return r2 < s2;
}

void orc_neighbors(const float *pm, const float *h, int64_t n, float kappa,
                   int mode, const int64_t *rows, int64_t k, int64_t *counts,
                   const int64_t *offs, int64_t *list)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < k; ++r) {
        int64_t i = rows[r], c = 0;
        for (int64_t j = 0; j < n; ++j) {
            if (j == i || !is_neighbour(pm, h, i, j, kappa, mode)) continue;
            if (list) list[offs[r] + c] = j;
            ++c;
        }
        counts[r] = c;
    }
}
