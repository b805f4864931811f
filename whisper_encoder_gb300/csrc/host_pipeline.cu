// wb_encode_host: the whole path from host audio to host hidden states (host code only).
//
// Batches are double-buffered on the device: while batch i computes on the caller's stream,
// batch i+1's audio uploads on one copy stream and batch i-1's output downloads on the other.
// Events tie each device buffer's reuse to the work that last used it:
//   in_ready[k]  upload of the audio in buffer k done      -> compute may read it
//   in_free[k]   log-mel (its only reader) done            -> the next upload may overwrite it
//   out_ready[k] encoder output in buffer k written        -> its download may start
//   out_free[k]  download of buffer k done                 -> the next batch may overwrite it
#include <cuda_runtime.h>

#include "../../include/wb.h"

namespace {

struct Events {
  cudaEvent_t e[10] = {};
  int n = 0;
  bool create() {
    for (n = 0; n < 10; ++n)
      if (cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
  ~Events() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);   // released once the events complete
  }
};

#define WB_TRY(x)                               \
  do {                                          \
    const wb_status st_ = (x);                  \
    if (st_ != WB_OK) return st_;               \
  } while (0)
#define WB_CU(x)                                \
  do {                                          \
    if ((x) != cudaSuccess) return WB_ECUDA;    \
  } while (0)

}  // namespace

extern "C" wb_status wb_encode_host(const wb_host_pipeline* p, const float* const* host_audio, void* const* host_out,
                                    int n_batches, void* stream) {
  if (!p || n_batches < 0 || p->batch < 1 || p->samples_per_batch < 0) return WB_EINVAL;
  if (n_batches == 0) return WB_OK;
  if (!host_audio || !host_out || !p->stem || !p->layers || !p->ln_post) return WB_EINVAL;
  const bool overlap = p->upload_stream != nullptr;
  if (overlap != (p->download_stream != nullptr)) return WB_EINVAL;
  const int nbuf = overlap ? 2 : 1;
  for (int k = 0; k < nbuf; ++k)
    if (!p->dev_audio[k] || !p->dev_out[k]) return WB_EINVAL;
  if (!p->dev_mel || !p->dev_x0) return WB_EINVAL;
  for (int i = 0; i < n_batches; ++i)
    if (!host_audio[i] || !host_out[i]) return WB_EINVAL;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t up = overlap ? static_cast<cudaStream_t>(p->upload_stream) : s;
  cudaStream_t down = overlap ? static_cast<cudaStream_t>(p->download_stream) : s;
  const size_t in_bytes = static_cast<size_t>(p->samples_per_batch) * sizeof(float);
  const size_t out_bytes = static_cast<size_t>(p->batch) * 1500 * static_cast<size_t>(p->dims.d_model) * 2;

  Events ev;
  cudaEvent_t *in_ready = ev.e, *in_free = ev.e + 2, *out_ready = ev.e + 4, *out_free = ev.e + 6;
  cudaEvent_t start = ev.e[8], done = ev.e[9];
  if (overlap) {
    if (!ev.create()) return WB_ECUDA;
    start = ev.e[8];
    done = ev.e[9];
    // the copy streams start after everything already queued on `stream`
    WB_CU(cudaEventRecord(start, s));
    WB_CU(cudaStreamWaitEvent(up, start, 0));
    WB_CU(cudaStreamWaitEvent(down, start, 0));
  }
  for (int i = 0; i < n_batches; ++i) {
    const int k = overlap ? (i & 1) : 0;
    if (overlap && i >= 2) WB_CU(cudaStreamWaitEvent(up, in_free[k], 0));
    WB_CU(cudaMemcpyAsync(p->dev_audio[k], host_audio[i], in_bytes, cudaMemcpyHostToDevice, up));
    if (overlap) {
      WB_CU(cudaEventRecord(in_ready[k], up));
      WB_CU(cudaStreamWaitEvent(s, in_ready[k], 0));
      if (i >= 2) WB_CU(cudaStreamWaitEvent(s, out_free[k], 0));
    }
    WB_TRY(wb_logmel(p->dev_audio[k], p->samples_per_batch, p->chunk_stride, p->batch, p->dims.n_mels, p->dev_mel,
                     p->ws_mel, p->ws_mel_bytes, s));
    if (overlap) WB_CU(cudaEventRecord(in_free[k], s));
    WB_TRY(wb_conv_stem(p->dev_mel, p->batch, &p->dims, p->stem, p->dev_x0, p->ws_stem, p->ws_stem_bytes, s));
    WB_TRY(wb_encoder_forward(p->dev_x0, p->batch, &p->dims, p->layers, p->ln_post, &p->precision, 0,
                              p->dims.n_layers, 1, p->dev_out[k], p->ws_enc, p->ws_enc_bytes, s));
    if (overlap) {
      WB_CU(cudaEventRecord(out_ready[k], s));
      WB_CU(cudaStreamWaitEvent(down, out_ready[k], 0));
    }
    WB_CU(cudaMemcpyAsync(host_out[i], p->dev_out[k], out_bytes, cudaMemcpyDeviceToHost, down));
    if (overlap) WB_CU(cudaEventRecord(out_free[k], down));
  }
  if (overlap) {
    // later work on `stream` comes after the last download (and the last upload)
    WB_CU(cudaEventRecord(done, down));
    WB_CU(cudaStreamWaitEvent(s, done, 0));
    WB_CU(cudaEventRecord(start, up));
    WB_CU(cudaStreamWaitEvent(s, start, 0));
  }
  return WB_OK;
}
