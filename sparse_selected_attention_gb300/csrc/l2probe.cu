// libqsa_l2probe.so: a measuring aid, not part of the attention path.
//
// It measures how fast this GPU's L2 serves the attention's access pattern:
// 128-byte rows gathered by id from an L2-resident table, eight lanes per row
// and one 16-byte load per lane, over a grid that fills every SM.  The
// benchmark takes this rate as the denominator of the attention's L2
// roofline (lts bytes per launch over the launch time).
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void gather_rows_kernel(const uint4 *__restrict__ table, long long table_rows,
                                   const int *__restrict__ rows, long long nids, unsigned *__restrict__ sink) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long groups = ((long long)gridDim.x * blockDim.x) >> 3;
    const int sub = threadIdx.x & 7;
    unsigned acc = 0u;
    for (long long i = tid >> 3; i < nids; i += groups) {
        const long long r = min(max((long long)__ldg(rows + i), 0ll), table_rows - 1);  // any id stays in the table
        const uint4 v = __ldcg(table + r * 8 + sub);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    sink[tid] = acc;  // keeps the loads
}

}  // namespace

// table: table_rows rows of 128 bytes (16-byte aligned); rows: nids row ids;
// sink: blocks * 256 words.  Returns a cudaError_t value (0 on success).
extern "C" int qsa_l2_gather_probe(const void *table, long long table_rows, const int *rows, long long nids,
                                   unsigned *sink, int blocks, void *stream) {
    if (!table || !rows || !sink || table_rows < 1 || nids < 0 || blocks < 1 ||
        (reinterpret_cast<uintptr_t>(table) & 15u) != 0)
        return (int)cudaErrorInvalidValue;
    gather_rows_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(static_cast<const uint4 *>(table), table_rows, rows,
                                                                  nids, sink);
    return (int)cudaGetLastError();
}
