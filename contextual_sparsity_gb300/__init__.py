"""GB300-native (sm_103a) decode-step hot path of Deja Vu contextual sparsity.

The compute path is the C-ABI library ``libdv.so`` (CUDA kernels for sm_103a);
``contextual_sparsity_gb300.dv`` is its thin Python binding. Importing this
package loads nothing: the binding loads the library on first use and raises if
it is missing (there is no CPU fallback).
"""
