// Tree-topology order: the spatial sort taken from an insertion-built tree.
//
// The GASPHiA tree-code page (section "排序算法") orders particles by the
// tree itself: read the leaves depth first and neighbours in the sequence
// are neighbours in space; parents hand their children disjoint ranges of
// the sort array, sized by the children's particle counts, from the top
// down.  Its tree is built by insertion (tree page after Burtscher &
// Pingali, sections "构建树结构" and "基于稠密存储的并行树构建实现方案"):
// every particle descends by octant, locks the child slot it needs with
// atomicCAS, and a slot already holding a particle is subdivided until the
// two separate; new nodes come from a global counter, so only the nodes in
// use are ever written (no clearing pass over a whole array).
//
// GB300 form, as an alternative to the radix sort of k_keys_sort.cu (same
// permutation, bit for bit):
//  * The octant at each depth is a 3-bit digit of the particle's Morton key
//    (x -> bit 0, y -> bit 1, z -> bit 2, the page's child numbering), so
//    the tree is the integer-cell tree whatever the insertion order.  Below
//    the key's last digit the particle's index supplies ten more digits:
//    every particle's digit string is unique, insertion always separates
//    two particles, and the depth-first order of the slots is the order of
//    (key, index) -- the stable sort.
//  * A slot holds EMPTY, LOCKED, a particle (-3 - index) or a node index.
//  * A cell is a node exactly when two or more rows share its digits, so the
//    cells of depths 1-4 are created before any insertion, from a histogram
//    of the keys' leading 12 bits (one block numbers them breadth first and
//    writes their slots).  Insertions then start at the deepest of these
//    nodes on their path, read from a directory indexed by the leading
//    digits: inserting into an empty tree instead makes every row contend
//    for the same few top-level slots while they are being split.
//    Only a slot holding a particle is locked (to subdivide it); an empty
//    slot is claimed with one compare-and-swap.  The lock holder writes the
//    new node (its eight slots, parent, the displaced particle) and
//    publishes the node index with a release store; others re-read
//    the slot (bounded: after kInsertLimit reads a particle gives up and
//    flags BH_ETIMEOUT).  A full node pool flags BH_ETREE_OVERFLOW.
//  * Counts bottom up without waiting: a node whose slots hold no nodes
//    computes its count and child offsets and climbs; at each parent an
//    arrival counter lets only the last child through, which then sums its
//    siblings (the same scheme as the centre-of-mass pass of k_build.cu).
//  * Placement: each particle descends its own path again, adding at every
//    node the offset of the slot it takes -- the start of that slot's range
//    inside the parent's.  The sum is its rank; the sorted key, index and
//    particle row are written there directly (the gather is fused).
#include <cuda_runtime.h>
#include <stdint.h>

#include "bh_internal.h"

namespace bh {

namespace {

constexpr int kEmpty = -1;
constexpr int kLocked = -2;
constexpr int kIndexDigits = 10;             // 3-bit digits of a < 2^30 index
constexpr unsigned kInsertLimit = 1u << 22;  // slot reads per particle
constexpr int kOrderThreads = 256;
constexpr int kDirDepth = 4;                 // depths created up front
constexpr int kDirSize = 8 + 64 + 512 + 4096;
constexpr int kTopThreads = 1024;

// Cells of depths 1..4 in breadth-first order: depth d starts at
// dir_base(d) and holds 8^d cells, indexed by the key's leading d digits.
__device__ __forceinline__ int dir_base(int d) {
  return d == 1 ? 0 : d == 2 ? 8 : d == 3 ? 72 : 584;
}

__device__ __forceinline__ int enc_particle(unsigned i) { return -3 - (int)i; }
__device__ __forceinline__ unsigned dec_particle(int c) { return (unsigned)(-3 - c); }

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release store: the writes before it (a new node's slots) are visible to
// any thread whose acquire load reads the stored value.
__device__ __forceinline__ void st_release(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// A row that could not be inserted: reported through the status word and
// remembered for this call's placement.
__device__ __forceinline__ void insert_failed(DevCtrl *c, unsigned code) {
  set_err(c, code);
  atomicExch(&c->step.order_fail, 1u);
}

// Octant digit of the depth-th level below the root (depth >= 1): Morton
// digits first, then the index's.
__device__ __forceinline__ int digit_at(unsigned long long key, unsigned idx, int depth,
                                        int bits) {
  if (depth <= bits) return (int)((key >> (3 * (bits - depth))) & 7ull);
  const int j = depth - bits - 1;
  return (int)((idx >> (3 * (kIndexDigits - 1 - j))) & 7u);
}

// Rows per depth-4 cell (the hist array is zeroed before the call).
__global__ void __launch_bounds__(kOrderThreads)
order_hist_kernel(const unsigned long long *keys, long long n, int bits, unsigned *hist) {
  __shared__ unsigned h[4096];
  for (int k = threadIdx.x; k < 4096; k += blockDim.x) h[k] = 0u;
  __syncthreads();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride)
    atomicAdd(&h[(int)(keys[i] >> (3 * (bits - kDirDepth)))], 1u);
  __syncthreads();
  for (int k = threadIdx.x; k < 4096; k += blockDim.x)
    if (h[k]) atomicAdd(&hist[k], h[k]);
}

// One block: the root and every cell of depths 1..4 holding two or more
// rows become nodes 0, 1, 2, ... in breadth-first order, with their slots
// pointing at their node children (EMPTY elsewhere: a cell of one row is
// claimed by that row's insertion); dir[] maps each cell to its node or -1.
__global__ void __launch_bounds__(kTopThreads)
order_top_kernel(const unsigned *hist, OrderBufs b, DevCtrl *ctrl) {
  __shared__ int cnt[kDirSize];
  __shared__ int part[kTopThreads];
  const int t = threadIdx.x;
  for (int k = t; k < 4096; k += kTopThreads) cnt[dir_base(4) + k] = (int)hist[k];
  __syncthreads();
  for (int d = 3; d >= 1; --d) {
    const int cells = 1 << (3 * d);
    for (int k = t; k < cells; k += kTopThreads) {
      int s = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) s += cnt[dir_base(d + 1) + 8 * k + c];
      cnt[dir_base(d) + k] = s;
    }
    __syncthreads();
  }
  // node numbers: 1 + rank among the cells with >= 2 rows (breadth first)
  constexpr int kPer = (kDirSize + kTopThreads - 1) / kTopThreads;
  const int lo = t * kPer, hi = min(lo + kPer, kDirSize);
  int mine = 0;
  for (int k = lo; k < hi; ++k) mine += cnt[k] >= 2;
  part[t] = mine;
  __syncthreads();
  for (int o = 1; o < kTopThreads; o <<= 1) {      // inclusive scan
    const int v = t >= o ? part[t - o] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  int rank = part[t] - mine;
  const int total = part[kTopThreads - 1];
  __syncthreads();
  for (int k = lo; k < hi; ++k) {   // cnt[] becomes the node number (or -1)
    const bool node = cnt[k] >= 2;
    cnt[k] = node ? 1 + rank : -1;
    rank += node;
  }
  __syncthreads();
  if (total + 1 > b.cap_nodes) {    // cannot happen: the pool holds 2n + 64
    if (t == 0) {
      atomicCAS(&ctrl->keep.err, 0u, kErrOverflow);
      ctrl->step.order_fail = 1u;
    }
    return;
  }
  for (int k = t; k < kDirSize; k += kTopThreads) b.dir[k] = cnt[k];
  if (t < 8) b.child[t] = cnt[t] >= 0 ? cnt[t] : kEmpty;      // the root
  if (t == 0) {
    b.parent[0] = -1;
    b.arrive[0] = 0;
    ctrl->step.trie_nodes = 1u + (unsigned)total;
  }
  for (int k = t; k < kDirSize; k += kTopThreads) {
    const int node = cnt[k];
    if (node < 0) continue;
    const int d = k < 8 ? 1 : k < 72 ? 2 : k < 584 ? 3 : 4;
    const int local = k - dir_base(d);
    b.parent[node] = d == 1 ? 0 : cnt[dir_base(d - 1) + (local >> 3)];
    b.arrive[node] = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int ch = d < kDirDepth ? cnt[dir_base(d + 1) + 8 * local + c] : -1;
      b.child[(long long)node * 8 + c] = ch >= 0 ? ch : kEmpty;
    }
  }
}

__global__ void __launch_bounds__(kOrderThreads)
order_insert_kernel(const unsigned long long *keys, long long n, int bits, OrderBufs b,
                    DevCtrl *ctrl) {
  // the top levels were not set up (pool too small): nothing to insert into
  if (*(volatile const unsigned *)&ctrl->step.order_fail) return;
  __shared__ int dir[kDirSize];
  for (int k = threadIdx.x; k < kDirSize; k += blockDim.x) dir[k] = b.dir[k];
  __syncthreads();
  const int max_depth = bits + kIndexDigits;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long key = keys[i];
    int node = 0, depth = 0;
#pragma unroll
    for (int d = kDirDepth; d >= 1; --d) {       // deepest node on the path
      const int v = dir[dir_base(d) + (int)(key >> (3 * (bits - d)))];
      if (v >= 0) {
        node = v;
        depth = d;
        break;
      }
    }
    unsigned reads = 0;
    for (;;) {
      if (++reads > kInsertLimit) {
        insert_failed(ctrl, kErrTimeout);
        break;
      }
      const int d1 = depth + 1;
      if (d1 > max_depth) {          // two equal digit strings: impossible
        insert_failed(ctrl, kErrOverflow);
        break;
      }
      int *slot = b.child + (long long)node * 8 + digit_at(key, (unsigned)i, d1, bits);
      const int c = ld_acquire(slot);
      if (c >= 0) {                  // a node: go down
        node = c;
        depth = d1;
        continue;
      }
      if (c == kEmpty) {
        if (atomicCAS(slot, kEmpty, enc_particle((unsigned)i)) == kEmpty) break;
        continue;
      }
      if (c == kLocked) {            // another particle is subdividing it
        __nanosleep(64);
        continue;
      }
      // the slot holds particle j: lock it, then split the cell
      if (atomicCAS(slot, c, kLocked) != c) continue;
      const unsigned j = dec_particle(c);
      const unsigned nn = atomicAdd(&ctrl->step.trie_nodes, 1u);
      if ((long long)nn >= b.cap_nodes || d1 + 1 > max_depth) {
        insert_failed(ctrl, kErrOverflow);
        atomicExch(slot, c);         // put j back; this particle stays out
        break;
      }
      int *nc = b.child + (long long)nn * 8;
#pragma unroll
      for (int k = 0; k < 8; ++k) nc[k] = kEmpty;
      b.parent[nn] = node;
      b.arrive[nn] = 0;
      nc[digit_at(keys[j], j, d1 + 1, bits)] = c;
      // the slot is locked by this thread: no other thread writes it, so a
      // release store publishes the node
      st_release(slot, (int)nn);
      node = (int)nn;
      depth = d1;
    }
  }
}

// Count and child offsets of node p from its slots (every node child's
// count already final).
__device__ __forceinline__ int settle(const OrderBufs &b, int p) {
  const int *ch = b.child + (long long)p * 8;
  int run = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = ld_acquire(ch + k);
    b.offs[(long long)p * 8 + k] = run;
    run += c >= 0 ? ld_acquire(b.count + c) : (c <= -3 ? 1 : 0);
  }
  b.count[p] = run;
  return run;
}

__global__ void __launch_bounds__(kOrderThreads)
order_nchild_kernel(OrderBufs b, const DevCtrl *ctrl) {
  long long total = ctrl->step.trie_nodes;
  if (total > b.cap_nodes) total = b.cap_nodes;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < total; p += stride) {
    const int4 *ch = reinterpret_cast<const int4 *>(b.child + p * 8);
    const int4 u = ch[0], v = ch[1];
    b.nchn[p] = (u.x >= 0) + (u.y >= 0) + (u.z >= 0) + (u.w >= 0) +
                (v.x >= 0) + (v.y >= 0) + (v.z >= 0) + (v.w >= 0);
  }
}

__global__ void __launch_bounds__(kOrderThreads)
order_count_kernel(OrderBufs b, DevCtrl *ctrl) {
  long long total = ctrl->step.trie_nodes;
  if (total > b.cap_nodes) total = b.cap_nodes;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; p0 < total;
       p0 += stride) {
    if (b.nchn[p0] != 0) continue;   // reached by its last arriving child
    int p = (int)p0;
    settle(b, p);
    // climb: only the last child to arrive at a parent goes on; a chain is
    // at most one step per depth
    for (int steps = 0; steps <= kMaxBits + kIndexDigits + 1; ++steps) {
      const int q = b.parent[p];
      if (q < 0) break;
      __threadfence();
      const int arrived = atomicAdd(&b.arrive[q], 1) + 1;
      if (arrived < b.nchn[q]) break;
      __threadfence();
      settle(b, q);
      p = q;
    }
  }
}

__global__ void __launch_bounds__(kOrderThreads)
order_place_kernel(const float4 *pm, const unsigned long long *keys, long long n, int bits,
                   OrderBufs b, unsigned long long *skeys, unsigned int *sidx, float4 *spm,
                   DevCtrl *ctrl) {
  const int max_depth = bits + kIndexDigits;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // After a failed insertion in this call the tree may miss rows; the
  // identity order then keeps every later stage on a permutation of valid
  // keys (the call's status already reports the failure).
  const bool failed = *(volatile const unsigned *)&ctrl->step.order_fail != 0u;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long key = keys[i];
    if (failed) {
      skeys[i] = key;
      sidx[i] = (unsigned)i;
      spm[i] = __ldg(pm + i);
      continue;
    }
    long long pos = 0;
    int node = 0;
    bool found = false;
    for (int d = 1; d <= max_depth; ++d) {
      const long long at = (long long)node * 8 + digit_at(key, (unsigned)i, d, bits);
      pos += b.offs[at];
      const int c = b.child[at];
      if (c >= 0 && c < b.cap_nodes) {
        node = c;
        continue;
      }
      found = c == enc_particle((unsigned)i);
      break;
    }
    if (!found || pos < 0 || pos >= n) {   // cannot happen after a clean insertion
      set_err(ctrl, kErrOverflow);
      continue;
    }
    skeys[pos] = key;
    sidx[pos] = (unsigned)i;
    spm[pos] = __ldg(pm + i);
  }
}

int grid_for(long long work, int num_sms) {
  long long blocks = (work + kOrderThreads - 1) / kOrderThreads;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_order_tree(const float4 *pm, const unsigned long long *keys, long long n,
                              int bits, OrderBufs &b, unsigned long long *skeys,
                              unsigned int *sidx, float4 *spm, DevCtrl *ctrl, int num_sms,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(b.hist, 0, 4096 * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int gp = grid_for(n, num_sms);
  order_hist_kernel<<<gp, kOrderThreads, 0, s>>>(keys, n, bits, b.hist);
  order_top_kernel<<<1, kTopThreads, 0, s>>>(b.hist, b, ctrl);
  order_insert_kernel<<<gp, kOrderThreads, 0, s>>>(keys, n, bits, b, ctrl);
  // the node passes stride up to the count the insertion left on the device
  long long nodes = n < b.cap_nodes ? n : b.cap_nodes;
  const int gn = grid_for(nodes, num_sms);
  order_nchild_kernel<<<gn, kOrderThreads, 0, s>>>(b, ctrl);
  order_count_kernel<<<gn, kOrderThreads, 0, s>>>(b, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_order_place(const float4 *pm, const unsigned long long *keys, long long n,
                               int bits, OrderBufs &b, unsigned long long *skeys,
                               unsigned int *sidx, float4 *spm, DevCtrl *ctrl, int num_sms,
                               cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  order_place_kernel<<<grid_for(n, num_sms), kOrderThreads, 0, s>>>(pm, keys, n, bits, b,
                                                                     skeys, sidx, spm, ctrl);
  return cudaGetLastError();
}

}  // namespace bh
