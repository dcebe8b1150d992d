// Speculative rollback of the per-sequence ring meta ("dory_msl.metal",
// cortiq-engine 0.8.57, kernel dory_o1_back): after a verify step has
// committed t draft rows and only some were accepted, each sequence's meta is
// rewound by the number of rejected rows.
//
// One rewind step of the page: a full window (win_len == W) keeps its length,
// its head steps back one slot (mod W) and far_len drops by one (32-bit
// unsigned); a window that is not full loses one key. A full window never
// leaves the full state, so n steps reduce to one closed form per branch,
// which is what the kernel applies. One thread per sequence.
#include "swa_internal.cuh"

namespace swa {

__global__ void rollback_kernel(swa_meta* __restrict__ meta, const int32_t* __restrict__ n_back,
                                int B, int cap, uint32_t* __restrict__ err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const swa_meta m = meta[b];
  bool bad = false;
  const SeqState st = sanitize_state(m, cap, &bad);
  const int n = n_back[b];
  if (bad || n < 0) {                       // leave a corrupt meta or request untouched
    set_err(err, SWA_DERR_META);
    return;
  }
  if (n == 0) return;
  swa_meta r = m;
  if (st.len0 == st.W) {
    const int back = n % st.W;
    r.win_head = (uint32_t)((st.head0 + st.W - back) % st.W);
    r.far_len = m.far_len - (uint32_t)n;    // modulo 2^32, as the page's uint arithmetic
  } else {
    if (n > st.len0) {                      // would drop below an empty window
      set_err(err, SWA_DERR_META);
      return;
    }
    r.win_len = (uint32_t)(st.len0 - n);
  }
  meta[b] = r;
}

int launch_rollback(swa_meta* meta, const int32_t* n_back, int B, int cap, uint32_t* err,
                    cudaStream_t s) {
  const int block = 128;
  rollback_kernel<<<(B + block - 1) / block, block, 0, s>>>(meta, n_back, B, cap, err);
  note_launch();
  return cuda_status(cudaGetLastError());
}

}  // namespace swa
