"""Seeded synthetic inputs for the TIDE reduce-scatter / all-gather hot path.

This package is shared by both sides of every parity check: the CPU oracle
(``oracle/``) and the CUDA library (``fsdp_layout_aware_gb300``).  It holds
none of the method's arithmetic -- no layout maps, no sums -- only

* ``gen``      counter-based random bits (SplitMix64) mapped to bf16 bit
               patterns, evaluated at arbitrary element indices on the host;
* ``configs``  the five workload descriptions (parameter shapes, N = M*L,
               value distributions) of the Llama-3.1-70B layer, the
               Qwen3-30B-A3B MoE layer, the Wan2.2 DiT block, the tiny
               hand-checkable group and the uneven/padding stress group;
* ``device``   a ctypes handle on ``libtide_synth.so``, the CUDA twin of
               ``gen`` that fills device buffers with the same bits.
"""
