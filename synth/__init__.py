"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds no arithmetic of the ZeRO-3 step: it draws random numbers
(Philox4x32-10), maps them to gradient / weight values, and describes the
parameter lists of the workloads.  Both the CPU oracle and the GPU harness
take their inputs from here, so that they see bit-identical data.

Modules
-------
philox     Philox4x32-10 counter-based generator (numpy), value mappings.
workloads  Parameter lists, rank counts and hyper-parameters of the workloads.
gpu        Fills device buffers with the same values (libzs_synth.so).
"""
