"""CPU oracle for CAAT-Net's partial channel-reduce -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The product library (``partial_activation_sync_gb300``) never does.
"""
