"""GB300 batch-1 decode megakernel: libamk.so (include/amk.h) and its binding.

``decode_megakernel_gb300.amk`` loads the CUDA library; importing the
package itself loads nothing, so the build step can run first.
"""
