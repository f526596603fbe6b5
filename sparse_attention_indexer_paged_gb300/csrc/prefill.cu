// Prefill over the paged cache (sparse_attn_indexer docs, the CPU indexer's
// prefill branch of forward_cpu).  A prefill chunk lays its requests' keys
// end to end (local_cu_seq_lens, B + 1 starts) and tags token row t with
// (ks, ke): ks is its request's start there, ke the end of the keys it sees.
// prefill_rows_kernel turns the tags into what the decode kernels take: the
// request of the row (the last start at or below ks) and its causal length
// ke - ks.  The rows then run through the decode schedule and logits kernels
// unchanged, grouped by request id and reading each request's block-table
// row through the row -> request map; no key is gathered or copied.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kPrefillThreads = 256;

__global__ void __launch_bounds__(kPrefillThreads)
    prefill_rows_kernel(const int32_t* __restrict__ ks, const int32_t* __restrict__ ke, int32_t num_rows,
                        const int32_t* __restrict__ starts, int32_t num_requests, int32_t* __restrict__ ctx,
                        int32_t* __restrict__ req, int32_t* status) {
  const int t = blockIdx.x * kPrefillThreads + threadIdx.x;
  if (t >= num_rows) return;
  const int32_t s = ks[t], e = ke[t];
  // number of starts <= s among starts[0 .. num_requests] (non-decreasing)
  int lo = 0, hi = num_requests + 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(starts + mid) <= s)
      lo = mid + 1;
    else
      hi = mid;
  }
  int r = lo - 1;
  r = r < 0 ? 0 : (r >= num_requests ? num_requests - 1 : r);
  int32_t len = e - s;
  if (len < 0) {
    if (status) atomicCAS(status, 0, DSA_ERR_INVALID_ARG);
    len = 0;
  }
  ctx[t] = len;
  req[t] = r;
}

}  // namespace

cudaError_t launch_prefill_rows(const int32_t* ks, const int32_t* ke, int32_t num_rows, const int32_t* starts,
                                int32_t num_requests, int32_t* ctx, int32_t* req, int32_t* status,
                                cudaStream_t stream) {
  const int grid = (num_rows + kPrefillThreads - 1) / kPrefillThreads;
  prefill_rows_kernel<<<grid, kPrefillThreads, 0, stream>>>(ks, ke, num_rows, starts, num_requests, ctx, req,
                                                            status);
  return cudaGetLastError();
}

}  // namespace dsa
