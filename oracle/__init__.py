"""CPU oracle for skip-softmax (BLASST) attention -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU baseline import this
package.  It shares no code with the CUDA library and does not import it.
"""
