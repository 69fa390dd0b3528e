// cf_cluster.cuh -- cluster collectives over distributed shared memory.
//
// ClusterReduce [CF §3.1.1, Alg. 1] and ClusterGather [CF §3.1.2, Alg. 2],
// page "ClusterFusion框架深度解析" (devpress.csdn.net), written for sm_103a:
//
//  * every round is a butterfly exchange with partner = rank ^ stride, where
//    rank is the block's rank inside its cluster (%cluster_ctarank);
//  * data is PUSHED: each thread writes its 16-byte pieces straight into the
//    partner's shared memory with st.async, which also signals the
//    partner's per-round mbarrier (complete_tx); the receiver waits on its
//    own mbarrier, so there is no cluster-wide barrier per round and threads
//    outside the collective (the TMA producer warp) never stall;
//  * each round of each collective owns its receive buffer and mbarrier, so a
//    buffer is written once per launch and no write-after-read hazard exists
//    between rounds (the page's double buffering, taken one step further).
//
// The collectives run on the NT consumer threads of a block, which
// synchronize with the named barrier kBar.  Every mbarrier is initialized
// with count 1 and armed once by the block itself (arrive.expect_tx with the
// byte count of its round) before the cluster's start barrier; it completes a
// single phase (parity 0) per launch.  All sizes are multiples of 4 floats.
#pragma once

#include "cf_ptx.cuh"

namespace cf {

struct OpSum {
  static __device__ __forceinline__ float apply(float a, float b) { return a + b; }
};
struct OpMax {
  static __device__ __forceinline__ float apply(float a, float b) { return fmaxf(a, b); }
};

// Bytes one round of each collective receives (what its mbarrier expects).
__host__ __device__ constexpr int allreduce_round_bytes(int n) { return n * 4; }
__host__ __device__ constexpr int reduce_scatter_round_bytes(int N, int r, int se) {
  return (N >> (r + 1)) * se * 4;
}
__host__ __device__ constexpr int gather_round_bytes(int r, int se) { return (1 << r) * se * 4; }

// Push n floats (n % 4 == 0) from local shared memory `src` to the same-offset
// location `dst_local` (an address in this block's window) of block `peer`,
// signalling that block's mbarrier at `bar_local`.
template <int NT>
__device__ __forceinline__ void push_to_peer(const float* src, const float* dst_local, int n,
                                             uint64_t* bar_local, uint32_t peer, int tid) {
  const uint32_t raddr = mapa(smem_u32(dst_local), peer);
  const uint32_t rbar = mapa(smem_u32(bar_local), peer);
  const float4* s4 = reinterpret_cast<const float4*>(src);
  for (int i = tid; i < n / 4; i += NT) st_async_v4(raddr + 16u * i, s4[i], rbar);
}

// ClusterReduce, all-reduce form (recursive doubling): afterwards every block
// holds op-reduced data[0..n).  rbuf holds log2(N) receive buffers of n
// floats; rbar log2(N) mbarriers.  The two operands of each round are
// combined as op(own, partner) -- for sum and max this equals
// op(partner, own) bit for bit, so all blocks finish with identical data.
template <class Op, int NT, int kBar>
__device__ void cluster_allreduce(float* data, int n, float* rbuf, uint64_t* rbar, int rank,
                                  int N, int tid, int* err) {
  int r = 0;
  for (int s = 1; s < N; s <<= 1, ++r) {
    float* rb = rbuf + r * n;
    push_to_peer<NT>(data, rb, n, &rbar[r], rank ^ s, tid);
    // Every thread has read its share of data for the push before any thread
    // overwrites data below: the threads that push nothing (n / 4 < NT) or
    // finish first would otherwise update chunks another thread has yet to
    // send, and the partner would add its own contribution twice.
    named_sync(kBar, NT);
    mbar_wait_cluster(&rbar[r], 0, err);
    for (int i = tid; i < n; i += NT) data[i] = Op::apply(data[i], rb[i]);
    named_sync(kBar, NT);
  }
}

// ClusterReduce with the online-softmax combine ([CF §3.2] 在线softmax; the
// page's ClusterReduce(max) followed by the rescaled ClusterReduce(sum), done
// in one butterfly).  data holds nrec records [o(D) | m | l | 2 pad] of
// partial attention states (m in log2 units, o unnormalized); afterwards every
// block holds, per record, m = max_c m_c, l = sum_c l_c 2^(m_c - m) and
// o = sum_c o_c 2^(m_c - m).  `scale` is 2*nrec floats of scratch.  Products
// and sums are rounded one by one (no fused multiply-add), so both sides of
// each exchange compute bit-identical records.
template <int NT, int kBar>
__device__ void cluster_allreduce_softmax(float* data, int nrec, int D, float* rbuf,
                                          uint64_t* rbar, float* scale, int rank, int N,
                                          int tid, int* err) {
  const int W = D + 4, n = nrec * W;
  int r = 0;
  for (int s = 1; s < N; s <<= 1, ++r) {
    float* rb = rbuf + r * n;
    push_to_peer<NT>(data, rb, n, &rbar[r], rank ^ s, tid);
    mbar_wait_cluster(&rbar[r], 0, err);
    for (int i = tid; i < nrec; i += NT) {
      const float ma = data[i * W + D], mb = rb[i * W + D];
      const float mm = fmaxf(ma, mb);
      scale[2 * i] = (mm == -INFINITY) ? 0.f : exp2f(ma - mm);
      scale[2 * i + 1] = (mm == -INFINITY) ? 0.f : exp2f(mb - mm);
    }
    named_sync(kBar, NT);
    for (int i = tid; i < n; i += NT) {
      const int rec = i / W, e = i - rec * W;
      if (e == D) {
        data[i] = fmaxf(data[i], rb[i]);
      } else if (e < D || e == D + 1) {
        data[i] = __fadd_rn(__fmul_rn(data[i], scale[2 * rec]), __fmul_rn(rb[i], scale[2 * rec + 1]));
      }
    }
    named_sync(kBar, NT);
  }
}

// ClusterReduce, reduce-scatter form (recursive halving, sum): data holds N
// slices of se floats; afterwards slice `rank` holds the cluster-wide sum of
// that slice (other slices are left partially reduced).  rbuf holds the
// rounds' receive buffers back to back ((N-1)*se floats in total).
template <int NT, int kBar>
__device__ void cluster_reduce_scatter(float* data, int se, float* rbuf, uint64_t* rbar,
                                       int rank, int N, int tid, int* err) {
  int lo = 0, r = 0;
  float* rb = rbuf;
  for (int s = N >> 1; s >= 1; s >>= 1, ++r) {
    const int keep = (rank & s) ? lo + s : lo;
    const int send = (rank & s) ? lo : lo + s;
    push_to_peer<NT>(data + send * se, rb, s * se, &rbar[r], rank ^ s, tid);
    mbar_wait_cluster(&rbar[r], 0, err);
    float* dst = data + keep * se;
    for (int i = tid; i < s * se; i += NT) dst[i] += rb[i];
    named_sync(kBar, NT);
    lo = keep;
    rb += s * se;
  }
}

// ClusterGather (recursive doubling, [CF §3.1.2]: the data moved per round
// doubles): data holds N slices of se floats of which slice `rank` is
// filled; afterwards every block holds all N slices.  Received blocks land
// directly in their final place in `data` (each slice is written once).
template <int NT, int kBar>
__device__ void cluster_gather(float* data, int se, uint64_t* gbar, int rank, int N, int tid,
                               int* err) {
  int r = 0;
  for (int s = 1; s < N; s <<= 1, ++r) {
    const int blk = rank & ~(s - 1);
    push_to_peer<NT>(data + blk * se, data + blk * se, s * se, &gbar[r], rank ^ s, tid);
    mbar_wait_cluster(&gbar[r], 0, err);
  }
  named_sync(kBar, NT);
}

// ---------------------------------------------------------- pull forms --
// In the pull forms a block reads its peers' shared memory directly
// (ld.shared::cluster) once they have signalled that the data is complete,
// so no receive buffers are needed.  Each exchange uses one mbarrier per block,
// initialized with count N-1 and completed (parity 0) by the peers'
// release-arrivals.

// Tell every other block of the cluster that this block's data for an
// exchange is complete: a cluster-scope release fence restricted to shared
// memory, then one relaxed arrival on the same-offset mbarrier `bar` of each
// peer.  Called by one thread after the producing threads have synchronized
// with it through a CTA barrier; the fence is cumulative, so it also orders
// their shared-memory writes before the peers' acquiring waits.  (A release
// arrival would order all of the thread's memory traffic and measured
// 0.8-2.5 us per call while the TMA stream runs.)
__device__ __forceinline__ void cluster_signal_peers(uint64_t* bar, int rank, int N) {
  const uint32_t b = smem_u32(bar);
  fence_release_smem_cluster();
  for (int q = 1; q < N; ++q) mbar_remote_arrive_relaxed(mapa(b, (uint32_t)((rank + q) % N)));
}

// ClusterReduce, reduce-scatter form by pulling [CF §3.1.1]: data holds N
// slices of n floats (n % 4 == 0) in every block; afterwards slice `rank` of
// this block holds the sum of slice `rank` over all blocks.  Slices other than
// `rank` are only read (by their owners), so they stay valid.  Each thread
// keeps four remote loads in flight per peer before it adds them.
template <int NT>
__device__ void cluster_pull_reduce_slice(float* data, int n, uint64_t* bar, int rank, int N,
                                          int tid, int* err) {
  constexpr int U = 4;
  mbar_wait_cluster(bar, 0, err);
  float4* own = reinterpret_cast<float4*>(data + (size_t)rank * n);
  const uint32_t base = smem_u32(own);
  const int n4 = n / 4;
  for (int i0 = tid; i0 < n4; i0 += NT * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * NT < n4) v[u] = own[i0 + u * NT];
    for (int q = 1; q < N; ++q) {
      const uint32_t rb = mapa(base, (uint32_t)((rank + q) % N));
      float4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * NT < n4) w[u] = ld_dsmem_f4(rb + 16u * (uint32_t)(i0 + u * NT));
#pragma unroll
      for (int u = 0; u < U; ++u) {
        v[u].x += w[u].x;
        v[u].y += w[u].y;
        v[u].z += w[u].z;
        v[u].w += w[u].w;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * NT < n4) own[i0 + u * NT] = v[u];
  }
}

// ClusterGather by pulling [CF §3.1.2]: block q's slice is `npieces` pieces
// of `nbytes` bytes (a multiple of 16) at buf + k * piece_stride + q * stride
// (k < npieces) in every block; afterwards every block holds all N slices.
// Each thread keeps four remote loads in flight before it stores them.
template <int NT>
__device__ void cluster_pull_gather(uint8_t* buf, int nbytes, int stride, int npieces,
                                    int piece_stride, uint64_t* bar, int rank, int N, int tid,
                                    int* err) {
  constexpr int U = 4;
  mbar_wait_cluster(bar, 0, err);
  const int n16 = nbytes / 16, per_peer = npieces * n16, total = (N - 1) * per_peer;
  for (int i0 = tid; i0 < total; i0 += NT * U) {
    uint4 w[U];
    uint8_t* dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = i0 + u * NT;
      if (idx < total) {
        const int peer = (rank + 1 + idx / per_peer) % N;
        const int rem = idx % per_peer;
        dst[u] = buf + (size_t)(rem / n16) * piece_stride + (size_t)peer * stride + 16 * (rem % n16);
        w[u] = ld_dsmem_u4(mapa(smem_u32(dst[u]), (uint32_t)peer));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * NT < total) *reinterpret_cast<uint4*>(dst[u]) = w[u];
  }
}

}  // namespace cf
