"""Speculative tree verification on GB300: tree-masked attention, acceptance and the online-training
loss, as hand-written sm_103a CUDA kernels behind a C ABI (libsv.so)."""
