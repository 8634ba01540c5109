// wd_routing.cuh - per-CTA routing tables in shared memory, built from the
// B*K expert ids of the call: which experts are routed to (ascending), and for
// each of them the list of (token, slot) indices s = b*K + k routed to it.
//
// This is metadata only (at most kStreamMaxSlots ints per list): activations
// are never copied or reordered, and each CTA builds its own copy, so no
// kernel launch or global buffer is added.  Every list is in ascending slot
// order, so all CTAs agree on it: work items that split one expert's list into
// chunks are handed to different CTAs and must partition it identically.
#pragma once

#include <stdint.h>

#include "wd_launch.h"

namespace wd {

struct RoutingTables {
  uint32_t* mask;  // [128]   bit e set if expert e is routed to (E <= 4096)
  int* wbase;      // [128]   number of routed experts in the words before
  int* expert;     // [S]     routed experts, ascending
  int* cnt;        // [S]     slots per routed expert (fill cursor while building)
  int* off;        // [S + 1] start of each expert's slot list in `slots`
  int* coff;       // [S + 1] start of each expert's chunks of `chunk` slots
  int* slots;      // [S]     slot lists, concatenated
  int* chunk_u;    // [S]     routed-expert index of each chunk
  int* ids;        // [S]     copy of the call's expert ids
  int* scalar;     // [0] routed experts U, [1] chunks, [2] 1 if an id was out of range
};

__host__ __device__ constexpr int routing_table_bytes() {
  return 4 * (128 + 128 + kStreamMaxSlots * 7 + 2 + 8);
}

__device__ __forceinline__ RoutingTables routing_tables_at(void* base) {
  constexpr int S = kStreamMaxSlots;
  int* p = static_cast<int*>(base);
  RoutingTables t;
  t.mask = reinterpret_cast<uint32_t*>(p);
  t.wbase = p + 128;
  t.expert = t.wbase + 128;
  t.cnt = t.expert + S;
  t.off = t.cnt + S;
  t.coff = t.off + S + 1;
  t.slots = t.coff + S + 1;
  t.chunk_u = t.slots + S;
  t.ids = t.chunk_u + S;
  t.scalar = t.ids + S;
  return t;
}

__device__ __forceinline__ void warp_exclusive_scan(int v, int& excl, int& total) {
  const int lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  excl = incl - v;
  total = __shfl_sync(0xFFFFFFFFu, incl, 31);
}

__device__ __forceinline__ int routed_index(const RoutingTables& t, int e) {
  return t.wbase[e >> 5] + __popc(t.mask[e >> 5] & ((1u << (e & 31)) - 1u));
}

// Build the tables with all `nthreads` threads of the CTA (contains
// __syncthreads; every thread must call it).  `chunk` is the number of slots
// per chunk (work items split an expert's token list into chunks).  Every
// phase but the two short scans is spread over all threads: the lists are
// filled through shared-memory atomics in any order, then each slot moves to
// its rank among its list's slots (found through `chunk_u`, which is filled
// last), so the lists end in ascending slot order whatever the order of the
// atomics.
__device__ __forceinline__ void build_routing_tables(const RoutingTables& t,
                                                     const int32_t* __restrict__ ids, int BK,
                                                     int E, int chunk, int nthreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwords = (E + 31) >> 5;
  for (int i = tid; i < nwords; i += nthreads) t.mask[i] = 0u;
  for (int i = tid; i < kStreamMaxSlots; i += nthreads) t.cnt[i] = 0;
  for (int s = tid; s < BK; s += nthreads) t.ids[s] = __ldg(ids + s);  // the only global reads
  if (tid == 0) t.scalar[2] = 0;
  __syncthreads();
  for (int s = tid; s < BK; s += nthreads) {
    const int e = t.ids[s];
    if (e >= 0 && e < E)
      atomicOr(&t.mask[e >> 5], 1u << (e & 31));
    else
      t.scalar[2] = 1;
  }
  __syncthreads();
  // routed experts before each mask word
  if (warp == 0) {
    int base = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const uint32_t word = (w0 + lane < nwords) ? t.mask[w0 + lane] : 0u;
      int excl, total;
      warp_exclusive_scan(__popc(word), excl, total);
      if (w0 + lane < nwords) t.wbase[w0 + lane] = base + excl;
      base += total;
    }
    if (lane == 0) t.scalar[0] = base;
  }
  __syncthreads();
  // the routed experts in ascending order, and each one's slot count
  for (int e = tid; e < E; e += nthreads)
    if (t.mask[e >> 5] & (1u << (e & 31))) t.expert[routed_index(t, e)] = e;
  for (int s = tid; s < BK; s += nthreads) {
    const int e = t.ids[s];
    if (e >= 0 && e < E) atomicAdd(&t.cnt[routed_index(t, e)], 1);
  }
  __syncthreads();
  const int U = t.scalar[0];
  if (warp == 0) {
    int base = 0, cbase = 0;
    for (int u0 = 0; u0 < U; u0 += 32) {
      const int u = u0 + lane;
      const int c = (u < U) ? t.cnt[u] : 0;
      const int nch = (c + chunk - 1) / chunk;
      int excl, total, cexcl, ctotal;
      warp_exclusive_scan(c, excl, total);
      warp_exclusive_scan(nch, cexcl, ctotal);
      if (u < U) {
        t.off[u] = base + excl;
        t.coff[u] = cbase + cexcl;
        t.cnt[u] = 0;  // becomes the fill cursor
      }
      base += total;
      cbase += ctotal;
    }
    if (lane == 0) {
      t.off[U] = base;
      t.coff[U] = cbase;
      t.scalar[1] = cbase;
    }
  }
  __syncthreads();
  // each slot takes a place in its expert's list, in any order ...
  for (int s = tid; s < BK; s += nthreads) {
    const int e = t.ids[s];
    if (e >= 0 && e < E) {
      const int u = routed_index(t, e);
      t.slots[t.off[u] + atomicAdd(&t.cnt[u], 1)] = s;
    }
  }
  __syncthreads();
  // ... then its rank in ascending slot order: the list's slots below it
  for (int s = tid; s < BK; s += nthreads) {
    const int e = t.ids[s];
    int pos = -1;
    if (e >= 0 && e < E) {
      const int u = routed_index(t, e);
      const int* l = t.slots + t.off[u];
      const int n = t.off[u + 1] - t.off[u];
      int r = 0;
      for (int i = 0; i < n; ++i) r += l[i] < s;
      pos = t.off[u] + r;
    }
    t.chunk_u[s] = pos;  // scratch: where slot s goes
  }
  __syncthreads();
  for (int s = tid; s < BK; s += nthreads) {
    const int pos = t.chunk_u[s];
    if (pos >= 0) t.slots[pos] = s;
  }
  __syncthreads();
  // the chunks of each routed expert's list
  for (int u = tid; u < U; u += nthreads) {
    const int nch = (t.off[u + 1] - t.off[u] + chunk - 1) / chunk;
    for (int q = 0; q < nch; ++q) t.chunk_u[t.coff[u] + q] = u;
  }
  __syncthreads();
}

}  // namespace wd
