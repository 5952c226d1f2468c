"""GB300-native stacked LSTM / GRU / tanh-RNN forward and backward-through-time.

The compute path is librnn.so (CUDA kernels for sm_103a behind a C-ABI,
include/rnn.h); ``rnn`` is its ctypes binding, ``build`` compiles it,
``synth`` draws the seeded synthetic inputs, ``runner`` allocates the
caller-owned buffers with PyTorch and drives one training or inference step.
"""
