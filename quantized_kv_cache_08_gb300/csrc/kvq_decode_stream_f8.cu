// The stream-K split kernel for FP8 E4M3 caches: kvq_decode_stream.cu built
// with its E4M3 code (stream_kernel_f8 and launch_split_stream_f8).  A
// separate translation unit keeps the q8_0 / q5_1 kernel's code unchanged.
#define KVQ_STREAM_F8 1
#include "kvq_decode_stream.cu"
