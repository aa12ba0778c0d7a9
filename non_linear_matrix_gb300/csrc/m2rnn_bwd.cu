// m2rnn_bwd.cu -- backward entry points (kernel under construction).
#include <cstddef>

#include "m2rnn.h"

extern "C" {

size_t m2rnn_bwd_workspace_size(const m2rnn_shape* s, int ckpt_given) {
  (void)s;
  (void)ckpt_given;
  return 0;
}

int m2rnn_bwd(const m2rnn_shape* s, const void*, const void*, const void*, const void*,
              const void*, const void*, const float*, const float*, const void*, const float*,
              float*, float*, float*, float*, float*, float*, float*, void*, size_t, void*) {
  (void)s;
  return M2RNN_ERR_UNSUPPORTED_SHAPE;
}

}  // extern "C"
