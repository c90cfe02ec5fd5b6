// Device-side KV page bookkeeping shared by the prepare, commit and reset
// kernels.  The sequence state (length, page count, page table, free-page
// bitmap) lives on the device so a round needs no host round trip.
//
// Pending-token invariant (Lecture 6 "Optimizing Autoregressive Decode",
// section 6.2): the cache holds the committed sequence minus its last token.
// A round writes the window at slots L..L+W-1; committing n accepted drafts sets
// the length to L + 1 + n, and pages wholly beyond the new length return to the
// pool (section 11: paged rollback edits the block-table length and frees the
// extra blocks).  Allocation takes the lowest free page index first.
#pragma once

#include "common.cuh"

namespace spec {

// Lowest free page via a warp-wide scan of the bitmap (bit set = free); marks it
// used.  Must be called by all 32 lanes of one warp; returns -1 if none.
SPEC_DEVICE_INLINE int warp_alloc_page(uint32_t* free_bits, int num_pages) {
  const int lane = threadIdx.x & 31;
  const int nwords = (num_pages + 31) >> 5;
  int found = -1;
  for (int w0 = 0; w0 < nwords && found < 0; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t bits = w < nwords ? free_bits[w] : 0u;
    const unsigned ballot = __ballot_sync(0xffffffffu, bits != 0u);
    if (ballot) {
      const int lw = __ffs(ballot) - 1;
      const uint32_t wb = __shfl_sync(0xffffffffu, bits, lw);
      found = (w0 + lw) * 32 + (__ffs(wb) - 1);
    }
  }
  if (found >= num_pages) found = -1;
  if (found >= 0 && lane == 0) free_bits[found >> 5] &= ~(1u << (found & 31));
  __syncwarp();
  return found;
}

// Give sequence s pages covering slots [0, upto).  Warp-cooperative.  Returns false
// (nothing half-done is rolled back) when the pool runs dry.
SPEC_DEVICE_INLINE bool warp_ensure_pages(int s, int upto, int32_t* seq_npages, int32_t* page_table, int max_pages,
                                          uint32_t* free_bits, int num_pages) {
  const int lane = threadIdx.x & 31;
  const int need = (upto + kPage - 1) / kPage;
  int npg = seq_npages[s];
  bool ok = need <= max_pages;
  while (ok && npg < need) {
    const int pg = warp_alloc_page(free_bits, num_pages);
    if (pg < 0) {
      ok = false;
      break;
    }
    if (lane == 0) page_table[(long long)s * max_pages + npg] = pg;
    ++npg;
  }
  if (lane == 0) seq_npages[s] = npg;
  __syncwarp();
  return ok;
}

// Return pages keep.. of sequence s to the pool (page table entries -1).  Single thread.
SPEC_DEVICE_INLINE void release_pages_from(int s, int keep, int32_t* seq_npages, int32_t* page_table, int max_pages,
                                           uint32_t* free_bits) {
  const int npg = seq_npages[s];
  for (int i = keep; i < npg; ++i) {
    const int pg = page_table[(long long)s * max_pages + i];
    if (pg >= 0) atomicOr(&free_bits[pg >> 5], 1u << (pg & 31));
    page_table[(long long)s * max_pages + i] = -1;
  }
  if (npg > keep) seq_npages[s] = keep;
}

// Set the cached length of sequence s and free every page whose first slot is
// >= new_len.  Single thread.
SPEC_DEVICE_INLINE void truncate_seq(int s, int new_len, int32_t* seq_len, int32_t* seq_npages, int32_t* page_table,
                                     int max_pages, uint32_t* free_bits) {
  release_pages_from(s, (new_len + kPage - 1) / kPage, seq_npages, page_table, max_pages, free_bits);
  seq_len[s] = new_len;
}

}  // namespace spec
