"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This package makes inputs only: hidden states, routings, scale banks and
compact expert banks.  It holds none of the decode path's arithmetic (no
activation quantizer, no block dot, no epilogue) and imports neither the
oracle nor the CUDA library.

Two kinds of expert bank are made:

  * converted banks (``banks.convert_*``): fp32 weights drawn from N(0, 0.02)
    and written into the bank formats the way an offline checkpoint converter
    would (ModelOpt-style NVFP4 with a per-projection weight_scale_2, a simple
    min/max Q4_K encoder, bf16 rounding).  Used where the bank fits in host
    memory and the value distribution matters.
  * counter-based banks (``counter``): every byte drawn from SplitMix64 at a
    counter equal to the byte's word index, then masked so that scale fields
    hold finite values of a realistic size.  The same bank can be produced on
    the GPU (torch integer ops) and, for any sub-range, on the host (numpy),
    so full-size banks of tens of GiB are filled on the device while the
    oracle regenerates just the experts it checks.
"""
