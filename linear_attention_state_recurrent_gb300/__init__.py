"""KDA (Kimi Delta Attention) gated delta-rule recurrence on GB300.

The compute lives in `libkda.so` (hand-written sm_103a CUDA behind a C ABI,
declared in include/kda.h); `kda` is its thin ctypes binding. Importing the
package loads nothing: `from linear_attention_state_recurrent_gb300 import kda`
loads the library and fails loudly if it has not been built.
"""
